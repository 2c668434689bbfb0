"""Seeded random shapes for the fused projection + RMSNorm + RoPE + band scatter,
every element against the oracle.

Each case draws the number of virtual ranks, local heads, batch, a ragged local
sequence, the layout, the RoPE pairing, the cluster form (two pairs sharing W, or
one pair) and the positions: the row index, or random rows of a table longer
than the sequence.  Outputs start poisoned (NaN), so every element must be
written; values must lie within max(2 bf16 ulp, 2e-2) of the oracle."""
import numpy as np
import pytest

import oracle
from ulysses_qkv_proj_gb300 import workloads as WL
from _util import assert_fused_close, to_dev_bf16, to_host_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from ulysses_qkv_proj_gb300 import binding as qb  # noqa: E402

N_CASES = 40


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_shape_against_oracle(seed):
    rng = np.random.default_rng(500 + seed)
    P = int(rng.choice([1, 2, 4, 8]))
    H_local = int(rng.integers(1, max(2, 12 // P) + 1))
    H = P * H_local
    B = int(rng.integers(1, 4))
    S = int(rng.integers(1, max(2, 1200 // (P * B)) + 1))
    layout = str(rng.choice(["bshd", "fused"]))
    rope = str(rng.choice(["rotate_half", "interleaved"]))
    flags = int(rng.choice([0, qb.FLAG_ONE_PAIR]))
    wl = WL.FusedWorkload(f"fuzz{seed}", P=P, B=B, S=S, num_heads=H, layout=layout, rope_style=rope)
    inp = WL.make_fused_inputs(wl)
    cos_sin, positions, pos_arg = inp.cos_sin, inp.positions, "given"
    if rng.random() < 0.5:
        n_pos = wl.S_global + int(rng.integers(1, 3000))
        cos_sin = WL.rope_table(n_pos)
        positions = rng.integers(0, n_pos, size=(P, B, S)).astype(np.int32)
    elif rng.random() < 0.5:
        pos_arg = None                       # positions = the token's row index
        positions = np.arange(wl.T, dtype=np.int32).reshape(P, B, S)
        cos_sin = WL.rope_table(wl.T)
    plan = qb.Plan(wl.hidden, H, P, layout, max_tokens=B * S, rope_style=rope, flags=flags)
    out = qb.alloc_outputs(plan, B, S)
    for t in out.values():
        t.view(torch.int16).fill_(-1)
    qb.qnre_forward(plan, to_dev_bf16(inp.x), to_dev_bf16(inp.w), to_dev_bf16(inp.q_norm_w),
                    to_dev_bf16(inp.k_norm_w), torch.from_numpy(cos_sin).cuda(),
                    None if pos_arg is None else torch.from_numpy(positions).cuda(), out)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    ref = oracle.qnre_forward(inp.x, inp.w, inp.q_norm_w, inp.k_norm_w, cos_sin, positions, P, H, layout, rope)
    for g in ref:
        assert_fused_close(to_host_f64(out[g]), ref[g], what=f"case {seed} ({P}x{B}x{S}, H={H}, {layout}, {rope})/{g}")
