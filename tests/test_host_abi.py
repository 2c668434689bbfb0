"""Host-side tests of the C ABI: the library loads, exports what include/qnre.h
declares, and rejects bad requests before touching the GPU (status codes only,
no compute call).  Runs without a GPU."""
import ctypes
import os
import subprocess
import sys

import pytest

from ulysses_qkv_proj_gb300 import binding as qb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(qb.LIB_PATH):
        from ulysses_qkv_proj_gb300 import build
        build.build()
    return qb.load_library()


def test_library_exports_every_declared_function(lib):
    names = qb.header_functions()
    assert set(names) >= {"qnre_plan_create", "qnre_plan_destroy", "qnre_forward", "ulysses_pack_head_chunk",
                          "ulysses_merge_output_head_chunk", "qnre_status_string", "qnre_plan_device_status"}
    out = subprocess.run(["nm", "-D", "--defined-only", qb.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)


def test_status_strings(lib):
    for code, name in qb.STATUS_NAMES.items():
        assert lib.qnre_status_string(code).decode().startswith(name)
    assert lib.qnre_status_string(99).decode() == "QNRE_ERR_UNKNOWN"


def _plan_create(lib, hidden=512, heads=4, head_dim=128, P=2, layout=0, max_tokens=64, rope=0, flags=0):
    h = ctypes.c_void_p()
    st = lib.qnre_plan_create(ctypes.byref(h), hidden, heads, head_dim, P, layout, max_tokens, rope, flags)
    return st, h


@pytest.mark.parametrize("kw,want", [
    (dict(head_dim=64), 2),             # head_dim fixed at 128: unsupported
    (dict(head_dim=0), 1),
    (dict(hidden=500), 1),              # hidden != heads * 128
    (dict(heads=3, hidden=384, P=2), 1),  # heads % P != 0 (pages: ValueError)
    (dict(P=0), 1),
    (dict(layout=7), 1),
    (dict(rope=5), 1),
    (dict(flags=0x80), 1),
    (dict(flags=0x6), 1),               # W multicast and one pair per cluster together
    (dict(max_tokens=0), 1),
    (dict(max_tokens=1 << 31), 5),
])
def test_plan_create_rejects(lib, kw, want):
    st, h = _plan_create(lib, **kw)
    assert st == want
    assert not h.value


def test_plan_create_null_handle(lib):
    assert lib.qnre_plan_create(None, 512, 4, 128, 2, 0, 64, 0, 0) == 1


def test_forward_rejects_null_plan(lib):
    o = qb._Out(None, None, None, None)
    assert lib.qnre_forward(None, 1, 1, 16, 16, 16, 16, 16, 1, None, ctypes.byref(o), None) == 1


def test_destroy_null_is_ok(lib):
    assert lib.qnre_plan_destroy(None) == 0


def _t4(ptr, shape, stride, dtype=0):
    t = qb._Tensor4()
    t.data = ptr
    for i in range(4):
        t.shape[i] = shape[i]
        t.stride[i] = stride[i]
    t.dtype = dtype
    return t


def _contig(shape):
    st = [1] * 4
    for i in (2, 1, 0):
        st[i] = st[i + 1] * shape[i + 1]
    return st


BASE = 1 << 40  # fake device addresses: validation never dereferences them


def _pack(lib, q, k, v, W, off, cnt, out):
    return lib.ulysses_pack_head_chunk(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), W, off, cnt, out, None)


def test_pack_validation(lib):
    shp = [1, 8, 4, 128]
    st = _contig(shp)
    n = 8 * 4 * 128 * 2
    q, k, v = (_t4(BASE + i * n, shp, st) for i in range(3))
    out = BASE + 3 * n
    assert _pack(lib, q, k, v, 3, 0, 1, out) == 1          # H % W != 0
    assert _pack(lib, q, k, v, 2, 1, 2, out) == 1          # offset + count > H_local
    assert _pack(lib, q, k, v, 2, -1, 1, out) == 1
    assert _pack(lib, q, k, v, 2, 0, 0, out) == 1
    assert _pack(lib, q, k, v, 0, 0, 1, out) == 1
    assert _pack(lib, q, k, v, 2, 0, 1, None) == 1
    k2 = _t4(BASE + n, [1, 8, 4, 64], _contig([1, 8, 4, 64]))
    assert _pack(lib, q, k2, v, 2, 0, 1, out) == 1         # shapes differ
    v2 = _t4(BASE + 2 * n, shp, st, dtype=1)
    assert _pack(lib, q, k, v2, 2, 0, 1, out) == 1         # dtypes differ
    q0 = _t4(BASE, shp, [st[0], st[1], 0, 1])
    assert _pack(lib, q0, k, v, 2, 0, 1, out) == 1         # stride 0 (not positive)
    q9 = _t4(BASE, shp, st, dtype=9)
    assert _pack(lib, q9, q9, q9, 2, 0, 1, out) == 2       # unknown dtype
    qa = _t4(BASE + 1, shp, st)
    assert _pack(lib, qa, k, v, 2, 0, 1, out) == 3         # misaligned for bf16
    assert _pack(lib, q, k, v, 2, 0, 1, out + 1) == 3
    assert _pack(lib, q, k, v, 2, 0, 1, BASE + n + 256) == 4  # out inside k's storage
    assert _pack(lib, q, k, v, 2, 0, 1, BASE - 256) == 4      # out runs into q


def test_pack_empty_is_ok_without_launch(lib):
    shp = [1, 0, 4, 128]
    st = [512, 512, 128, 1]
    q = _t4(BASE, shp, st)
    assert _pack(lib, q, q, q, 2, 0, 1, BASE + (1 << 20)) == 0


def test_merge_validation(lib):
    shp = [1, 8, 2, 128]
    st = _contig(shp)
    r = _t4(BASE, shp, st)
    out = BASE + (1 << 20)
    m = lib.ulysses_merge_output_head_chunk
    assert m(ctypes.byref(r), 3, 2, 0, out, None) == 1     # 2 % 3 != 0
    assert m(ctypes.byref(r), 2, 2, 2, out, None) == 1     # offset + count > local_heads
    assert m(ctypes.byref(r), 2, 0, 0, out, None) == 1
    assert m(ctypes.byref(r), 2, 2, -1, out, None) == 1
    assert m(ctypes.byref(r), 2, 2, 0, None, None) == 1
    assert m(ctypes.byref(r), 2, 2, 0, BASE + 64, None) == 4  # out overlaps received
    assert m(ctypes.byref(r), 2, 2, 0, out + 1, None) == 3
    re_ = _t4(BASE, [1, 0, 2, 128], st)
    assert m(ctypes.byref(re_), 2, 2, 0, out, None) == 0   # empty call


def test_oracle_not_imported_by_product():
    """The product path never imports the oracle (fresh interpreter)."""
    code = ("import sys; sys.path.insert(0, %r); import ulysses_qkv_proj_gb300.binding, "
            "ulysses_qkv_proj_gb300.workloads; print('oracle' in sys.modules or "
            "any(m.startswith('oracle.') for m in sys.modules))") % ROOT
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True)
    assert res.stdout.strip() == "False", res.stderr


def test_product_sources_do_not_reference_oracle():
    pkg = os.path.join(ROOT, "ulysses_qkv_proj_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f


def test_sage2_workspace_bytes(lib):
    n = ctypes.c_uint64()
    assert lib.ulysses_sage2_workspace_bytes(2, 1, 300, 4, 128, ctypes.byref(n)) == 0
    chunks = 2   # 300 rows per rank in chunks of 256
    assert n.value == (2 * 2 * chunks * 1 * 4 * 128 + 2 * 1 * 4 * 128) * 4
    assert lib.ulysses_sage2_workspace_bytes(2, 1, 300, 4, 96, ctypes.byref(n)) == 2    # D not 64 / 128
    assert lib.ulysses_sage2_workspace_bytes(3, 1, 300, 4, 128, ctypes.byref(n)) == 1   # H % P
    assert lib.ulysses_sage2_workspace_bytes(2, 1, 0, 4, 128, ctypes.byref(n)) == 1
    assert lib.ulysses_sage2_workspace_bytes(2, 1, 65535 * 32 + 1, 4, 128, ctypes.byref(n)) == 5
    assert lib.ulysses_sage2_workspace_bytes(2, 1, 300, 4, 128, None) == 1


def test_sage2_scatter_validation(lib):
    """Every call here fails a host check, so nothing is launched (fake addresses)."""
    P, B, L, H, D = 2, 1, 64, 4, 128
    shp = [P * B, L, H, D]
    st = _contig(shp)
    n = P * B * L * H * D * 2
    q, k, v = (_t4(BASE + i * n, shp, st) for i in range(3))
    o = BASE + (1 << 30)
    ws_n = ctypes.c_uint64()
    assert lib.ulysses_sage2_workspace_bytes(P, B, L, H, D, ctypes.byref(ws_n)) == 0
    mb = 1 << 20
    outs = [o, o + 8 * mb, o + 16 * mb, o + 24 * mb, o + 25 * mb, o + 26 * mb, o + 27 * mb]

    def call(q=q, k=k, v=v, P=P, U=P * L, outs=outs, ws=ws_n.value):
        return lib.ulysses_sage2_scatter_qkv(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), P, U, *outs, ws,
                                             None)
    assert call(U=0) == 1
    assert call(U=P * L + 1) == 1
    assert call(P=3) == 1                                      # P does not divide the batch extent
    assert call(ws=ws_n.value - 1) == 5                        # workspace too small
    assert call(outs=outs[:6] + [None]) == 1
    assert call(outs=[o + 8] + outs[1:]) == 3                  # q_out not 16-byte aligned
    assert call(outs=outs[:2] + [o + 16 * mb + 4] + outs[3:]) == 3
    assert call(outs=[BASE + 256] + outs[1:]) == 4             # q_out inside q
    assert call(outs=outs[:1] + [o + 64] + outs[2:]) == 4      # k_out overlaps q_out
    assert call(outs=outs[:6] + [o + 24 * mb]) == 4            # workspace overlaps q_scale
    f32 = _t4(BASE, shp, st, dtype=2)
    assert call(q=f32, k=f32, v=f32) == 2                      # fp32 inputs are not served
    k16 = _t4(BASE + n, shp, st, dtype=1)
    assert call(k=k16) == 1                                    # mixed dtypes
    k96 = _t4(BASE + n, [P * B, L, H, 96], _contig([P * B, L, H, 96]))
    assert call(k=k96) == 1                                    # shapes differ
    q96 = _t4(BASE, [P * B, L, H, 96], _contig([P * B, L, H, 96]))
    assert call(q=q96, k=q96, v=q96) == 2                      # D = 96
    qs = _t4(BASE, shp, [st[0], st[1] + 4, st[2], 1])
    assert call(q=qs) == 3                                     # row stride not a multiple of 16 bytes
    qe = _t4(BASE, [P * B, 0, H, D], st)
    assert call(q=qe, k=qe, v=qe) == 1                         # an empty sequence has no statistics


def test_plan_reserve_sms_rejects_without_a_plan(lib):
    assert lib.qnre_plan_reserve_sms(None, 8) == 1


def test_schedule_calls_reject_before_launch(lib):
    """Every call here fails a host check, so nothing is launched (fake addresses)."""
    shp = [1, 8, 4, 128]
    st = _contig(shp)
    n = 8 * 4 * 128 * 2
    q, k, v = (_t4(BASE + i * n, shp, st) for i in range(3))
    out = BASE + (1 << 20)
    I2 = ctypes.c_int * 2
    P2 = ctypes.c_void_p * 2
    pack = lib.ulysses_pack_head_chunk_schedule
    args = (ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), 2)
    assert pack(*args, 0, I2(0, 1), I2(1, 1), P2(out, out + n), None) == 1          # no chunks
    assert pack(*args, 9, (ctypes.c_int * 9)(), (ctypes.c_int * 9)(), (ctypes.c_void_p * 9)(), None) == 5
    assert pack(*args, 2, None, I2(1, 1), P2(out, out + n), None) == 1              # NULL array
    assert pack(*args, 2, I2(0, 1), I2(1, 1), P2(out, out + 256), None) == 4        # outputs overlap
    assert pack(*args, 2, I2(0, 1), I2(1, 2), P2(out, out + n), None) == 1          # chunk 2 past H_local
    r = _t4(BASE, [1, 8, 2, 128], _contig([1, 8, 2, 128]))
    merge = lib.ulysses_merge_output_head_chunk_schedule
    R2 = ctypes.POINTER(qb._Tensor4) * 2
    views = R2(ctypes.pointer(r), ctypes.pointer(r))
    assert merge(views, 2, 2, 2, I2(0, 0), out, None) == 1                           # the same band twice
    assert merge(views, 2, 2, 0, I2(0, 1), out, None) == 1
    assert merge(None, 2, 2, 2, I2(0, 1), out, None) == 1


def test_plan_describe_rejects_without_a_plan(lib):
    info = qb._PlanInfo()
    assert lib.qnre_plan_describe(None, 1, 1, ctypes.byref(info)) == 1


def test_debug_bounds_release_build_is_unsupported(lib):
    n = ctypes.c_ulonglong(7)
    assert lib.qnre_debug_bounds(ctypes.byref(n), 0) == 2  # QNRE_ERR_UNSUPPORTED: no checks compiled in
    assert n.value == 0
    assert lib.qnre_debug_bounds(None, 0) == 1


def test_debug_build_exports_every_declared_function():
    """libqnre_debug.so (QNRE_DEBUG_BOUNDS=1) builds from the same sources and
    serves the same ABI; without a GPU its count query fails with QNRE_ERR_CUDA."""
    from ulysses_qkv_proj_gb300 import build
    path = build.build(debug_bounds=True)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in qb.header_functions():
        assert n in exported, n
    dbg = ctypes.CDLL(path)
    dbg.qnre_debug_bounds.restype = ctypes.c_int
    dbg.qnre_debug_bounds.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), ctypes.c_int]
    assert dbg.qnre_debug_bounds(None, 0) == 1
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except ImportError:
        has_gpu = False
    if not has_gpu:
        n = ctypes.c_ulonglong(0)
        assert dbg.qnre_debug_bounds(ctypes.byref(n), 0) == 6


def test_scatter_qkv_alias_covers_every_destination_band(lib):
    """out [P, B, P*S, head_count, 3D] is P times one source band: an input that
    overlaps only the last destination rank's part of it is still an alias."""
    P, PB, S, H, D = 2, 2, 8, 4, 128
    shp = [PB, S, H, D]
    n = PB * S * H * D * 2
    q, k, v = (_t4(BASE + i * n, shp, _contig(shp)) for i in range(3))
    out_bytes = P * PB * S * 1 * 3 * D * 2
    out = BASE - out_bytes + 256                 # its last 256 bytes lie over q
    f = lib.ulysses_scatter_qkv_head_chunk
    assert f(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), P, 0, 1, out, None) == 4
    out = BASE - out_bytes // P - 256            # clear of q for one band only
    assert f(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), P, 0, 1, out, None) == 4
