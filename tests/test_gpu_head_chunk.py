"""GPU parity of the head-chunk pack and merge against the CPU oracle (bit-exact)."""
import numpy as np
import pytest

import oracle
from ulysses_qkv_proj_gb300 import workloads as WL
from _util import to_dev_bf16, to_host_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from ulysses_qkv_proj_gb300 import binding as qb  # noqa: E402


def _rand_bits(shape, seed, dtype=np.uint16):
    rng = np.random.default_rng(seed)
    if dtype == np.uint32:
        return rng.integers(0, 1 << 32, size=shape, dtype=np.uint64).astype(np.uint32)
    return rng.integers(0, 1 << 16, size=shape).astype(np.uint16)


def _dev(a, tdtype):
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).view(tdtype).cuda()
    return torch.from_numpy(a.view(np.int16)).view(tdtype).cuda()


def _host(t):
    t = t.contiguous().cpu()
    if t.element_size() == 4:
        return t.view(torch.int32).numpy().view(np.uint32)
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("B,S,H,D,W,sched", [
    (1, 37, 8, 128, 2, [(0, 1), (1, 2), (3, 1)]),      # ragged S, uneven schedule
    (2, 130, 12, 128, 3, [(0, 2), (2, 2)]),            # batch 2, W=3
    (1, 5, 4, 64, 4, [(0, 1)]),                        # H_local = 1
    (2, 33, 6, 128, 1, [(0, 3), (3, 3)]),              # world size 1
    (1, 300, 56, 128, 2, [(0, 7), (7, 14), (21, 7)]),  # the pages' uneven schedule shape
])
@pytest.mark.parametrize("tdtype", ["bf16", "fp16", "fp32"])
def test_pack_merge_strided_views(B, S, H, D, W, sched, tdtype):
    td = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[tdtype]
    npd = np.uint32 if tdtype == "fp32" else np.uint16
    buf = _rand_bits((B, S, 3, H, D), seed=B * 1000 + S, dtype=npd)
    tb = _dev(buf, td)
    q, k, v = tb[:, :, 0], tb[:, :, 1], tb[:, :, 2]   # positive-stride non-contiguous views
    L = H // W
    merged = {c: _dev(_rand_bits((B, S, H, D), seed=7, dtype=npd), td) for c in "qkv"}
    merged_ref = {c: _host(merged[c]) for c in "qkv"}
    for off, cnt in sched:
        out = torch.empty((B, S, W * cnt, 3 * D), dtype=td, device="cuda")
        qb.ulysses_pack_head_chunk(q, k, v, W, off, cnt, out)
        torch.cuda.synchronize()
        want = oracle.pack_head_chunk(buf[:, :, 0], buf[:, :, 1], buf[:, :, 2], W, off, cnt)
        assert np.array_equal(_host(out), want)
        for ci, c in enumerate("qkv"):
            rec = out[..., ci * D:(ci + 1) * D]            # strided received band
            qb.ulysses_merge_output_head_chunk(rec, W, L, off, merged[c])
            merged_ref[c] = oracle.merge_output_head_chunk(want[..., ci * D:(ci + 1) * D], W, L, off,
                                                           merged_ref[c])
    torch.cuda.synchronize()
    for ci, c in enumerate("qkv"):
        got = _host(merged[c])
        assert np.array_equal(got, merged_ref[c])
        if sum(cnt for _, cnt in sched) == L:   # a complete schedule reconstructs the input
            assert np.array_equal(got, buf[:, :, ci])


def test_pack_element_path_nonunit_inner_stride():
    """A view with a non-unit innermost stride takes the element path; still bit-exact."""
    B, S, H, D, W = 1, 19, 4, 128, 2
    big = _rand_bits((B, S, H, 2 * D), seed=3)
    tb = to_dev_bf16(big)
    q = tb[..., ::2]          # stride 2 along D
    k = tb[..., 1::2]
    v = tb[..., :D]           # unit stride (mixed paths in one call)
    out = torch.empty((B, S, W * 1, 3 * D), dtype=torch.bfloat16, device="cuda")
    qb.ulysses_pack_head_chunk(q, k, v, W, 1, 1, out)
    torch.cuda.synchronize()
    want = oracle.pack_head_chunk(big[..., ::2], big[..., 1::2], big[..., :D], W, 1, 1)
    assert np.array_equal(to_host_bits(out), want)


def test_merge_contiguous_received_leaves_rest_untouched():
    B, S, W, L, D = 2, 77, 4, 5, 128
    off, cnt = 2, 2
    rec = _rand_bits((B, S, W * cnt, D), seed=4)
    base = _rand_bits((B, S, W * L, D), seed=5)
    out = to_dev_bf16(base)
    qb.ulysses_merge_output_head_chunk(to_dev_bf16(rec), W, L, off, out)
    torch.cuda.synchronize()
    got = to_host_bits(out)
    assert np.array_equal(got, oracle.merge_output_head_chunk(rec, W, L, off, base))
    band = np.zeros(W * L, bool)
    for r in range(W):
        band[r * L + off: r * L + off + cnt] = True
    assert np.array_equal(got[:, :, ~band], base[:, :, ~band])


def test_pack_merge_on_side_stream():
    B, S, H, D, W = 1, 64, 8, 128, 2
    buf = _rand_bits((B, S, 3, H, D), seed=8)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        tb = to_dev_bf16(buf)
        out = torch.empty((B, S, W * 2, 3 * D), dtype=torch.bfloat16, device="cuda")
        qb.ulysses_pack_head_chunk(tb[:, :, 0], tb[:, :, 1], tb[:, :, 2], W, 1, 2, out, stream=s)
    s.synchronize()
    assert np.array_equal(to_host_bits(out),
                          oracle.pack_head_chunk(buf[:, :, 0], buf[:, :, 1], buf[:, :, 2], W, 1, 2))


def test_alias_rejected_on_device_tensors():
    tb = torch.zeros((1, 8, 3, 4, 128), dtype=torch.bfloat16, device="cuda")
    q, k, v = tb[:, :, 0], tb[:, :, 1], tb[:, :, 2]
    out = tb.view(-1)[: 8 * 2 * 384].view(1, 8, 2, 384)
    with pytest.raises(qb.QnreError) as e:
        qb.ulysses_pack_head_chunk(q, k, v, 2, 0, 1, out)
    assert e.value.status == 4


@pytest.mark.slow
def test_pages_headchunk_shape_full_size():
    """[1, 37760, 56, 128] over 2 virtual ranks with schedule [7, 14, 7], full size, bit-exact."""
    wl = WL.HEADCHUNK_WORKLOADS["headchunk_p2_s37760_h56"]
    buf = WL.make_headchunk_buffer(wl.B, wl.S_global, wl.num_heads)
    tb = to_dev_bf16(buf)
    W, L, D, S = wl.P, wl.H_local, wl.D, wl.S
    for r_s in range(wl.P):
        rows = slice(r_s * S, (r_s + 1) * S)
        q, k, v = tb[:, rows, 0], tb[:, rows, 1], tb[:, rows, 2]
        hq, hk, hv = buf[:, rows, 0], buf[:, rows, 1], buf[:, rows, 2]
        merged = torch.zeros((wl.B, S, wl.num_heads, D), dtype=torch.bfloat16, device="cuda")
        for off, cnt in wl.schedule:
            out = torch.empty((wl.B, S, W * cnt, 3 * D), dtype=torch.bfloat16, device="cuda")
            qb.ulysses_pack_head_chunk(q, k, v, W, off, cnt, out)
            qb.ulysses_merge_output_head_chunk(out[..., :D], W, L, off, merged)
            torch.cuda.synchronize()
            assert np.array_equal(to_host_bits(out), oracle.pack_head_chunk(hq, hk, hv, W, off, cnt))
        assert np.array_equal(to_host_bits(merged), hq)


@pytest.mark.parametrize("B,S,H,D,W,sched,tdtype", [
    (1, 300, 56, 128, 2, [(0, 7), (7, 14), (21, 7)], "bf16"),   # the pages' uneven schedule
    (2, 130, 12, 128, 3, [(0, 2), (2, 2)], "fp16"),
    (1, 37, 8, 64, 2, [(0, 1), (1, 2), (3, 1)], "fp32"),
])
def test_schedule_calls_match_single_calls(B, S, H, D, W, sched, tdtype):
    """The schedule forms (one launch each) equal the single-chunk calls made in
    order, and the oracle, bit for bit."""
    td = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[tdtype]
    npd = np.uint32 if tdtype == "fp32" else np.uint16
    buf = _rand_bits((B, S, 3, H, D), seed=S + W, dtype=npd)
    tb = _dev(buf, td)
    q, k, v = tb[:, :, 0], tb[:, :, 1], tb[:, :, 2]
    L = H // W
    outs = [torch.empty((B, S, W * cnt, 3 * D), dtype=td, device="cuda") for _, cnt in sched]
    qb.ulysses_pack_head_chunk_schedule(q, k, v, W, sched, outs)
    base = _rand_bits((B, S, H, D), seed=3, dtype=npd)
    merged = _dev(base, td)
    qb.ulysses_merge_output_head_chunk_schedule([o[..., :D] for o in outs], W, L, [off for off, _ in sched], merged)
    torch.cuda.synchronize()
    ref = base.copy()
    for (off, cnt), o in zip(sched, outs):
        want = oracle.pack_head_chunk(buf[:, :, 0], buf[:, :, 1], buf[:, :, 2], W, off, cnt)
        assert np.array_equal(_host(o), want)
        ref = oracle.merge_output_head_chunk(want[..., :D], W, L, off, ref)
    assert np.array_equal(_host(merged), ref)


def test_schedule_mixed_copy_units_and_rejections():
    B, S, H, D, W = 1, 40, 8, 128, 2
    buf = _rand_bits((B, S, 3, H, D), seed=11)
    tb = to_dev_bf16(buf)
    q, k, v = tb[:, :, 0], tb[:, :, 1], tb[:, :, 2]
    sched = [(0, 1), (1, 3)]
    # the second output starts 2 bytes into a buffer: that chunk takes the element path
    big = torch.empty((B * S * W * 3 * 3 * D + 8,), dtype=torch.bfloat16, device="cuda")
    o0 = torch.empty((B, S, W * 1, 3 * D), dtype=torch.bfloat16, device="cuda")
    o1 = big[1:1 + B * S * W * 3 * 3 * D].view(B, S, W * 3, 3 * D)
    qb.ulysses_pack_head_chunk_schedule(q, k, v, W, sched, [o0, o1])
    torch.cuda.synchronize()
    for (off, cnt), o in zip(sched, [o0, o1]):
        assert np.array_equal(to_host_bits(o), oracle.pack_head_chunk(buf[:, :, 0], buf[:, :, 1], buf[:, :, 2],
                                                                      W, off, cnt))
    out = torch.empty((B, S, W * 2, 3 * D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(qb.QnreError) as e:   # both chunks write the same buffer
        qb.ulysses_pack_head_chunk_schedule(q, k, v, W, [(0, 2), (2, 2)], [out, out])
    assert e.value.status == 4
    with pytest.raises(qb.QnreError) as e:
        qb.ulysses_pack_head_chunk_schedule(q, k, v, W, [(0, 1)] * 9, [out] * 9)
    assert e.value.status == 5
    merged = torch.zeros((B, S, H, D), dtype=torch.bfloat16, device="cuda")
    rec = out[..., :D]
    with pytest.raises(qb.QnreError) as e:   # bands [0, 2) and [1, 3) overlap
        qb.ulysses_merge_output_head_chunk_schedule([rec, rec], W, H // W, [0, 1], merged)
    assert e.value.status == 1
