"""GPU parity (bit-exact) of the ordinary and head-chunk exchange layouts over P virtual ranks."""
import numpy as np
import pytest

import oracle
from ulysses_qkv_proj_gb300 import workloads as WL
from _util import to_dev_bf16, to_host_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from ulysses_qkv_proj_gb300 import binding as qb  # noqa: E402

TD = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


def _bits(shape, seed, tdtype="bf16"):
    rng = np.random.default_rng(seed)
    if tdtype == "fp32":
        return rng.integers(0, 1 << 32, size=shape, dtype=np.uint64).astype(np.uint32)
    return rng.integers(0, 1 << 16, size=shape).astype(np.uint16)


def _dev(a, tdtype="bf16"):
    if a.dtype == np.uint32:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).view(TD[tdtype]).cuda()
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(TD[tdtype]).cuda()


def _host(t):
    t = t.contiguous().cpu()
    if t.element_size() == 4:
        return t.view(torch.int32).numpy().view(np.uint32)
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("P,B,S,H,D", [(1, 2, 7, 3, 128), (2, 1, 37, 8, 128), (4, 2, 33, 8, 64), (3, 1, 5, 6, 128)])
@pytest.mark.parametrize("tdtype", ["bf16", "fp32"])
def test_scatter_gather_heads(P, B, S, H, D, tdtype):
    x = _bits((P, B, S, H, D), seed=P * 100 + S, tdtype=tdtype)
    tx = _dev(x, tdtype)
    y = torch.empty((P, B, P * S, H // P, D), dtype=TD[tdtype], device="cuda")
    qb.ulysses_scatter_heads(tx, y)
    back = torch.empty_like(tx)
    qb.ulysses_gather_heads(y, back)
    torch.cuda.synchronize()
    assert np.array_equal(_host(y), oracle.scatter_heads(x))
    assert np.array_equal(_host(back), x)
    assert np.array_equal(_host(back), oracle.gather_heads(oracle.scatter_heads(x)))


def test_scatter_heads_rejects():
    x = torch.zeros((2, 1, 4, 3, 128), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((2, 1, 8, 1, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(qb.QnreError) as e:
        qb.ulysses_scatter_heads(x, y)  # 3 heads over 2 ranks
    assert e.value.status == 1
    with pytest.raises(qb.QnreError) as e:
        qb.ulysses_gather_heads(torch.zeros((2, 1, 5, 1, 128), dtype=torch.bfloat16, device="cuda"),
                                torch.empty((2, 1, 2, 2, 128), dtype=torch.bfloat16, device="cuda"))
    assert e.value.status == 1  # S_global 5 over 2 ranks


@pytest.mark.parametrize("B,S_g,cnt,D,W", [(1, 40, 3, 128, 2), (2, 36, 2, 128, 4), (1, 9, 1, 64, 3)])
def test_pack_output_sequence_chunk_strided(B, S_g, cnt, D, W):
    big = _bits((B, S_g, cnt + 2, D), seed=S_g)
    t = to_dev_bf16(big)
    x = t[:, :, 1:1 + cnt]  # a strided band of a wider output
    out = torch.empty((W, B, S_g // W, cnt, D), dtype=torch.bfloat16, device="cuda")
    qb.ulysses_pack_output_sequence_chunk(x, W, out)
    torch.cuda.synchronize()
    assert np.array_equal(to_host_bits(out), oracle.pack_output_sequence_chunk(big[:, :, 1:1 + cnt], W))


@pytest.mark.parametrize("P,B,S,L,bands", [
    (2, 1, 40, 7, [(0, 2), (2, 3), (5, 2)]),
    (4, 2, 17, 3, [(0, 1), (1, 2)]),
    (1, 1, 9, 4, [(0, 4)]),
])
def test_head_chunk_exchanges_match_oracle_and_ordinary(P, B, S, L, bands):
    H, D = P * L, 128
    buf = _bits((P * B, S, 3, H, D), seed=P * 10 + S)
    tb = to_dev_bf16(buf)
    q, k, v = tb[:, :, 0], tb[:, :, 1], tb[:, :, 2]
    qs = [buf[r * B:(r + 1) * B, :, 0] for r in range(P)]
    ks = [buf[r * B:(r + 1) * B, :, 1] for r in range(P)]
    vs = [buf[r * B:(r + 1) * B, :, 2] for r in range(P)]
    # input side
    for off, cnt in bands:
        out = torch.empty((P, B, P * S, cnt, 3 * D), dtype=torch.bfloat16, device="cuda")
        qb.ulysses_scatter_qkv_head_chunk(q, k, v, P, off, cnt, out)
        torch.cuda.synchronize()
        want = oracle.scatter_qkv_head_chunk(qs, ks, vs, off, cnt)
        assert np.array_equal(to_host_bits(out), np.stack(want))
    # output side: attention output bands [P, B, P*S, L, D] back to every rank's [B, S, H, D]
    o = _bits((P, B, P * S, L, D), seed=99)
    base = _bits((P, B, S, H, D), seed=98)
    outs = to_dev_bf16(base)
    ref = [base[r] for r in range(P)]
    for off, cnt in bands:
        band = np.ascontiguousarray(o[:, :, :, off:off + cnt])
        qb.ulysses_gather_output_head_chunk(to_dev_bf16(band), L, off, outs)
        ref = oracle.gather_output_head_chunk(list(band), L, off, ref)
    torch.cuda.synchronize()
    got = to_host_bits(outs)
    assert np.array_equal(got, np.stack(ref))
    if sum(c for _, c in bands) == L:
        assert np.array_equal(got, oracle.gather_heads(o))


@pytest.mark.slow
def test_pages_shape_ordinary_and_exchanges_full_size():
    """[1, 37760, 56, 128] over 2 virtual ranks: scatter/gather heads and both exchanges, bit-exact."""
    wl = WL.HEADCHUNK_WORKLOADS["headchunk_p2_s37760_h56"]
    P, S, H, D, L = wl.P, wl.S, wl.num_heads, wl.D, wl.H_local
    buf = WL.make_headchunk_buffer(1, wl.S_global, H, D)          # [1, S_g, 3, H, D]
    ranks = buf.reshape(P, S, 3, H, D)                             # rank r_s = rows [r_s*S, +S)
    q = np.ascontiguousarray(ranks[:, None, :, 0])                 # [P, 1, S, H, D]
    tq = to_dev_bf16(q)
    y = torch.empty((P, 1, P * S, L, D), dtype=torch.bfloat16, device="cuda")
    qb.ulysses_scatter_heads(tq, y)
    back = torch.empty_like(tq)
    qb.ulysses_gather_heads(y, back)
    torch.cuda.synchronize()
    want_y = oracle.scatter_heads(q)
    assert np.array_equal(to_host_bits(y), want_y)
    assert np.array_equal(to_host_bits(back), q)
    tb = to_dev_bf16(ranks)                                        # [P, S, 3, H, D] = [P*B, S, 3, H, D]
    outs = torch.zeros((P, 1, S, H, D), dtype=torch.bfloat16, device="cuda")
    for off, cnt in wl.schedule:
        pay = torch.empty((P, 1, P * S, cnt, 3 * D), dtype=torch.bfloat16, device="cuda")
        qb.ulysses_scatter_qkv_head_chunk(tb[:, :, 0], tb[:, :, 1], tb[:, :, 2], P, off, cnt, pay)
        # the received q band of every rank goes straight back through the output exchange
        band = pay[..., :D].contiguous()
        qb.ulysses_gather_output_head_chunk(band, L, off, outs)
        torch.cuda.synchronize()
        assert np.array_equal(to_host_bits(pay[..., :D]), want_y[:, :, :, off:off + cnt])
    assert np.array_equal(to_host_bits(outs), q)


def test_rows_beyond_one_grid_dimension():
    """More than 65535 x 128 sequence rows per segment: the copy's row blocks grow to
    256 rows so the grid's y extent stays within 65535 (16-byte head rows keep the
    arrays at about 0.5 GB)."""
    P, B, S, H, D = 2, 1, 65535 * 128 + 1000, 2, 8
    x = np.random.default_rng(5).integers(0, 1 << 16, size=(P, B, S, H, D), dtype=np.uint16)
    tx = _dev(x)
    y = torch.empty((P, B, P * S, H // P, D), dtype=torch.bfloat16, device="cuda")
    qb.ulysses_scatter_heads(tx, y)
    back = torch.empty_like(tx)
    qb.ulysses_gather_heads(y, back)
    torch.cuda.synchronize()
    assert np.array_equal(_host(y), oracle.scatter_heads(x))
    assert np.array_equal(_host(back), x)
