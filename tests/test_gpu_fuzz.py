"""Seeded randomized parity sweep over the whole call surface, against the fp64
oracle (GPU through the C ABI).

Each case draws, from its own seed: head_dim {64, 128, 256}, block size
{16, 32}, group size {1, 2, 4, 8, 16} and kv heads {1, 2, 4}, fp16 or bf16,
fp32 or q-dtype output, the softmax scale (1/sqrt(D) times 0.5..2), one query
token or 2..40 (so that a unit's rows fall below, at and past the 16 rows of
the warp-level kernel and the 128-row tiles of the tcgen05 kernel), a ragged
batch with empty, one-token and block-aligned sequences, spare table columns
and pool blocks, sometimes a masked table entry (-1 or an id past the pool),
the entry point (single pass, split-KV, multi-token) with a partition mode
(automatic, one pass, an explicit size, balanced), and the kernel choice
(library's own, or either multi-token kernel forced), sometimes a
max_context_len above every length, up to past the table's reach, and for
some split-KV cases the allocation-free entry point.  Output
and workspace start as NaN, so a row or partial that nothing wrote shows; the
workspace has exactly the size the library reports.

Bar: max |gpu - oracle| <= 2e-3 on fp32 output; q-dtype output within 2e-3
plus one ulp of the oracle rounded to that dtype; no device error.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_08_gb300 as pa

pytestmark = pytest.mark.gpu

TOL = 2e-3
DEV = "cuda:0"
N_CASES = 192


def draw(seed):
    g = np.random.default_rng(1000 + seed)
    c = dict(D=int(g.choice([64, 128, 256])), bs=int(g.choice([16, 32])),
             G=int(g.choice([1, 2, 4, 8, 16])), Hkv=int(g.choice([1, 2, 4])),
             dtype=[torch.float16, torch.bfloat16][int(g.integers(2))])
    c["q_len"] = 1 if g.random() < 0.5 else int(g.integers(2, 41))
    c["B"] = int(g.integers(1, 7)) if c["q_len"] == 1 else int(g.integers(1, 4))
    tmax = 1200 if c["q_len"] == 1 else 400
    lens = []
    for _ in range(c["B"]):
        kind = g.random()
        if kind < 0.1:
            lens.append(0)
        elif kind < 0.2:
            lens.append(1)
        elif kind < 0.3:
            lens.append(c["bs"] * int(g.integers(1, 9)))
        else:
            lens.append(int(g.integers(1, tmax)))
    c["lens"] = lens
    c["mb_extra"] = int(g.integers(0, 3))
    c["spare"] = int(g.integers(0, 6))
    c["mask"] = ["none", "minus_one", "past_pool"][int(g.choice(3, p=[0.7, 0.15, 0.15]))]
    c["entry"] = ("multi" if c["q_len"] > 1 else
                  ["single", "splitkv", "multi"][int(g.choice(3, p=[0.2, 0.6, 0.2]))])
    c["pt"] = ["auto", "one", "split", "balanced"][int(g.choice(4, p=[0.4, 0.15, 0.3, 0.15]))]
    c["split_pages"] = int(g.integers(1, 9))
    c["out_q"] = bool(g.random() < 0.2)
    c["scale_mul"] = float(g.uniform(0.5, 2.0))
    c["kernel"] = ["auto", "mma", "tile"][int(g.choice(3, p=[0.6, 0.2, 0.2]))]
    c["mask_seed"] = int(g.integers(1 << 30))
    # sometimes a max_context_len above every length (a serving loop passing
    # the model's limit), up to past the table's reach
    c["ctx_extra"] = int(g.integers(1, 3 * 32 * 12)) if g.random() < 0.2 else 0
    # split-KV calls: sometimes through the allocation-free entry point
    c["noalloc"] = bool(g.random() < 0.3)
    return c


def make_inputs(seed, c):
    gen = torch.Generator().manual_seed(2000 + seed)
    B, Q, D, bs, Hkv = c["B"], c["q_len"], c["D"], c["bs"], c["Hkv"]
    H = c["G"] * Hkv
    pages = [(t + bs - 1) // bs for t in c["lens"]]
    mb = max(1, max(pages)) + c["mb_extra"]
    pool = max(1, sum(pages) + c["spare"])
    perm = torch.randperm(pool, generator=gen)
    bt = torch.full((B, mb), -1, dtype=torch.int32)
    k = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[k:k + n].to(torch.int32)
        k += n
    used = [b for b, n in enumerate(pages) if n > 0]
    if c["mask"] != "none" and used:
        g = np.random.default_rng(c["mask_seed"])
        b = used[int(g.integers(len(used)))]
        j = int(g.integers(pages[b]))
        bt[b, j] = -1 if c["mask"] == "minus_one" else pool + int(g.integers(0, 4))
    dt = c["dtype"]
    q = torch.randn(B, Q, H, D, generator=gen).to(dt)
    kc = torch.randn(pool, bs, Hkv, D, generator=gen).to(dt)
    vc = torch.randn(pool, bs, Hkv, D, generator=gen).to(dt)
    lens = torch.tensor(c["lens"], dtype=torch.int32)
    return q, kc, vc, bt, lens, c["scale_mul"] / math.sqrt(D), max(c["lens"]) + c["ctx_extra"]


def partition_tokens(c, max_ctx):
    bs = c["bs"]
    if c["pt"] == "auto":
        return 0
    if c["pt"] == "one":
        return max(1, -(-max_ctx // bs)) * bs
    if c["pt"] == "split":
        return c["split_pages"] * bs
    return pa.PARTITION_BALANCED


def nan_workspace(nbytes):
    """Exactly the reported size; 0xFF bytes read as NaN in every fp32 partial."""
    return torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=DEV)


def check(got, want, out_q, dtype):
    g = got.double().cpu().numpy()
    assert np.isfinite(g).all(), "non-finite output"
    if not out_q:
        err = np.abs(g - want).max()
        assert err <= TOL, f"max abs err {err:.3e} > {TOL}"
        return
    want_r = torch.from_numpy(want).to(dtype).double().numpy()
    a = np.abs(want_r)
    mant = 10 if dtype == torch.float16 else 7
    ulp = np.where(a > 0, 2.0 ** (np.floor(np.log2(np.where(a > 0, a, 1.0))) - mant), 2.0 ** -24)
    bad = np.abs(g - want_r) > TOL + ulp
    assert not bad.any(), f"{int(bad.sum())} elements beyond 2e-3 + 1 ulp"


@pytest.mark.parametrize("seed", range(N_CASES), ids=lambda s: f"case{s}")
def test_random_case_vs_oracle(seed, switches):
    c = draw(seed)
    switches(kernel=c["kernel"])
    q, kc, vc, bt, lens, scale, max_ctx = make_inputs(seed, c)
    if c["q_len"] == 1 and c["entry"] != "multi":
        want = oracle.decode(q[:, 0].contiguous(), kc, vc, bt, lens, scale)
    else:
        want = oracle.decode_multi(q, kc, vc, bt, lens, scale)
    qd, kd, vd, btd, ld = (t.to(DEV) for t in (q, kc, vc, bt, lens))
    out_dtype = c["dtype"] if c["out_q"] else torch.float32
    pt = partition_tokens(c, max_ctx)
    if c["entry"] == "multi":
        out = torch.full(qd.shape, float("nan"), dtype=out_dtype, device=DEV)
        ws = nan_workspace(pa.workspace_size_multi(qd, kd, btd, out_dtype, max_ctx, pt))
        pa.decode_multi(out, qd, kd, vd, btd, ld, scale, max_ctx, pt, workspace=ws)
    else:
        q1 = qd[:, 0].contiguous()
        out = torch.full(q1.shape, float("nan"), dtype=out_dtype, device=DEV)
        need = pa.workspace_size(q1, kd, btd, out_dtype, max_ctx, pt)
        if c["entry"] == "single":
            pa.decode(out, q1, kd, vd, btd, ld, scale)
        elif c["noalloc"] and need <= 8 << 20:
            pa.decode_splitkv_noalloc(out, q1, kd, vd, btd, ld, scale, max_ctx, pt)
        else:
            ws = nan_workspace(pa.workspace_size(q1, kd, btd, out_dtype, max_ctx, pt))
            pa.decode_splitkv(out, q1, kd, vd, btd, ld, scale, max_ctx, pt, workspace=ws)
    torch.cuda.synchronize()
    check(out, want, c["out_q"], c["dtype"])
    assert pa.device_error() == 0
