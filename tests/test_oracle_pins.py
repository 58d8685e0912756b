"""Pins for the fp64 oracle, each against something other than the oracle itself.

A plausible slip anywhere in the oracle (a dropped scale, a wrong GQA head map,
t % bs and t // bs swapped, K and V swapped, no max subtraction, -1 read as a
Python index, a bad fp16/bf16 decode) fails at least one test here:

  - hand-worked closed forms (tests/golden/hand_worked_cases.json)
  - a single attended token returns that token's V row exactly
  - equal keys return the mean of V
  - one dominant score (far beyond exp's range) returns that token's V row
  - a dense fp64 brute force written independently below
  - torch's scaled_dot_product_attention in fp64 for an identity table
  - invariance under permuting the physical pool with the table remapped
  - masking readings: -1 / out-of-range entries, clamping to the table row,
    poison in unreferenced memory
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from paged_kv_attention_08_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_cases.json")


def _t(x, dtype):
    return torch.tensor(x, dtype=torch.float64).to(dtype)


# --------------------------------------------------------------------------
# independent dense brute force (numpy / scipy), written from the definition
# --------------------------------------------------------------------------
def brute_force(q, k_cache, v_cache, block_tables, context_lens, scale):
    """Gather each sequence densely, then softmax(q K^T * scale) V per head."""
    qd = q.to(torch.float64).numpy()
    kd = k_cache.to(torch.float64).numpy()
    vd = v_cache.to(torch.float64).numpy()
    bt = np.asarray(block_tables, dtype=np.int64)
    lens = np.asarray(context_lens, dtype=np.int64)
    B, H, D = qd.shape
    NB, bs, Hkv, _ = kd.shape
    G = H // Hkv
    out = np.zeros((B, H, D))
    for b in range(B):
        n = min(max(int(lens[b]), 0), bt.shape[1] * bs)
        toks = np.arange(n)
        ent = bt[b, toks // bs] if n else np.zeros(0, dtype=np.int64)
        ok = (ent >= 0) & (ent < NB)
        toks, ent = toks[ok], ent[ok]
        if toks.size == 0:
            continue
        Kb = kd[ent, toks % bs]            # [n, Hkv, D]
        Vb = vd[ent, toks % bs]
        for h in range(H):
            s = scale * (Kb[:, h // G, :] @ qd[b, h])
            out[b, h] = scipy.special.softmax(s) @ Vb[:, h // G, :]
    return out


def small_case(seed, B, H, Hkv, D, bs, lens, dtype=torch.float16, spare=3):
    """Random small problem with a shuffled pool and `spare` unreferenced blocks."""
    g = torch.Generator().manual_seed(seed)
    pages = [(t + bs - 1) // bs for t in lens]
    mb = max(1, max(pages))
    pool = sum(pages) + spare
    perm = torch.randperm(pool, generator=g)
    bt = torch.full((B, mb), -1, dtype=torch.int32)
    c = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[c:c + n].to(torch.int32)
        c += n
    q = torch.randn(B, H, D, generator=g).to(dtype)
    k = torch.randn(pool, bs, Hkv, D, generator=g).to(dtype)
    v = torch.randn(pool, bs, Hkv, D, generator=g).to(dtype)
    return q, k, v, bt, torch.tensor(lens, dtype=torch.int32), 1.0 / math.sqrt(D)


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------
@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_hand_worked_golden(case):
    q = _t(case["q"], torch.float16)
    k = _t(case["k_cache"], torch.float16)
    v = _t(case["v_cache"], torch.float16)
    out = oracle.decode(q, k, v, case["block_tables"], case["context_lens"], case["scale"])
    np.testing.assert_allclose(out, np.array(case["expected"]), rtol=0, atol=1e-15)


def test_hand_worked_file_is_what_its_script_writes():
    """The stored closed-form cases are exactly what the committed script
    builds from the logistic function (no oracle, no GPU involved)."""
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "make_hand_worked_cases", os.path.join(os.path.dirname(GOLDEN), "make_hand_worked_cases.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    assert json.load(open(GOLDEN)) == mod.build()


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_single_token_returns_its_v_row(dtype):
    q, k, v, bt, _, scale = small_case(1, B=3, H=8, Hkv=2, D=16, bs=4, lens=[5, 9, 2], dtype=dtype)
    lens = torch.tensor([1, 1, 1], dtype=torch.int32)
    # V rows carry awkward values: subnormals, extremes, signed zero
    if dtype == torch.float16:
        special = torch.tensor([6e-8, -6e-8, 65504.0, -65504.0, -0.0, 1e-5, 3.14159, -2.5])
    else:
        special = torch.tensor([1e-38, -9e-39, 3.0e38, -3.0e38, -0.0, 1e-5, 3.14159, -2.5])
    v.view(-1)[: special.numel()] = special.to(dtype)
    v[int(bt[0, 0]), 0, 0, :8] = special.to(dtype)
    out = oracle.decode(q, k, v, bt, lens, scale)
    G = 8 // 2
    for b in range(3):
        for h in range(8):
            want = v[int(bt[b, 0]), 0, h // G].to(torch.float64).numpy()
            np.testing.assert_array_equal(out[b, h], want)


def test_equal_keys_give_mean_of_v():
    q, k, v, bt, lens, scale = small_case(2, B=2, H=4, Hkv=2, D=8, bs=4, lens=[7, 13])
    k[:] = k[0, 0, 0]                 # every key row equal -> all scores equal
    out = oracle.decode(q, k, v, bt, lens, scale)
    vd = v.to(torch.float64).numpy()
    for b, n in enumerate([7, 13]):
        rows = [vd[int(bt[b, t // 4]), t % 4] for t in range(n)]   # [n][Hkv][D]
        mean = np.mean(np.stack(rows), axis=0)
        for h in range(4):
            np.testing.assert_allclose(out[b, h], mean[h // 2], rtol=0, atol=1e-12)


def test_dominant_score_selects_its_row():
    # scores of several hundred: exp without the max subtraction overflows to inf
    q, k, v, bt, lens, scale = small_case(3, B=1, H=2, Hkv=1, D=64, bs=8, lens=[30])
    q[:] = 8.0
    j = 17
    k[int(bt[0, j // 8]), j % 8, 0, :] = 8.0          # s_j = 64 * 64 / 8 = 512
    out = oracle.decode(q, k, v, bt, lens, scale)
    want = v[int(bt[0, j // 8]), j % 8, 0].to(torch.float64).numpy()
    for h in range(2):
        np.testing.assert_allclose(out[0, h], want, rtol=1e-15, atol=1e-300)


# --------------------------------------------------------------------------
# independent implementations
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("shape", [
    dict(B=2, H=8, Hkv=2, D=16, bs=4, lens=[9, 16]),
    dict(B=3, H=6, Hkv=3, D=8, bs=2, lens=[1, 5, 12]),
    dict(B=1, H=4, Hkv=4, D=32, bs=16, lens=[47]),
    dict(B=2, H=16, Hkv=1, D=8, bs=8, lens=[31, 3]),
])
def test_matches_dense_bruteforce(shape, dtype):
    q, k, v, bt, lens, scale = small_case(4, dtype=dtype, **shape)
    got = oracle.decode(q, k, v, bt, lens, scale)
    want = brute_force(q, k, v, bt, lens, float(np.float32(scale)))
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_matches_torch_sdpa_identity_table():
    B, H, Hkv, D, bs, T = 1, 8, 2, 32, 4, 37
    nb = (T + bs - 1) // bs
    g = torch.Generator().manual_seed(5)
    q = torch.randn(B, H, D, generator=g).to(torch.float16)
    k = torch.randn(nb, bs, Hkv, D, generator=g).to(torch.float16)
    v = torch.randn(nb, bs, Hkv, D, generator=g).to(torch.float16)
    bt = torch.arange(nb, dtype=torch.int32)[None]
    scale = float(np.float32(1.0 / math.sqrt(D)))
    got = oracle.decode(q, k, v, bt, [T], scale)
    K = k.to(torch.float64).reshape(nb * bs, Hkv, D)[:T].permute(1, 0, 2).repeat_interleave(H // Hkv, 0)
    V = v.to(torch.float64).reshape(nb * bs, Hkv, D)[:T].permute(1, 0, 2).repeat_interleave(H // Hkv, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.to(torch.float64)[0][:, None, :], K, V, scale=scale)[:, 0, :]
    np.testing.assert_allclose(got[0], ref.numpy(), rtol=0, atol=1e-12)


def test_pool_permutation_invariance():
    q, k, v, bt, lens, scale = small_case(6, B=3, H=8, Hkv=2, D=16, bs=4, lens=[10, 3, 16], spare=5)
    base = oracle.decode(q, k, v, bt, lens, scale)
    g = torch.Generator().manual_seed(7)
    NB = k.shape[0]
    perm = torch.randperm(NB, generator=g)          # new position of old block i is perm[i]
    k2, v2 = torch.empty_like(k), torch.empty_like(v)
    k2[perm], v2[perm] = k, v
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0).long()].to(torch.int32), bt)
    moved = oracle.decode(q, k2, v2, bt2, lens, scale)
    np.testing.assert_array_equal(moved, base)


def test_workload_tiny_matches_bruteforce():
    x = workloads.make("tiny", seed=0)
    got = oracle.decode(x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens, x.scale)
    want = brute_force(x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens,
                       float(np.float32(x.scale)))
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    rows = np.array([[1, 31], [0, 0], [1, 4]])
    np.testing.assert_array_equal(
        oracle.decode_rows(x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens, x.scale, rows),
        got[rows[:, 0], rows[:, 1]])


# --------------------------------------------------------------------------
# masking readings
# --------------------------------------------------------------------------
def test_masked_entries_are_excluded():
    q, k, v, bt, lens, scale = small_case(8, B=2, H=4, Hkv=2, D=8, bs=4, lens=[16, 12], spare=2)
    NB = k.shape[0]
    bt_bad = bt.clone()
    bt_bad[0, 1] = -1          # in-range unallocated entry
    bt_bad[1, 2] = NB + 5      # out-of-range id
    got = oracle.decode(q, k, v, bt_bad, lens, scale)
    want = brute_force(q, k, v, bt_bad, lens, float(np.float32(scale)))
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    # the same as dropping those tokens: sequence 0 keeps pages 0,2,3; sequence 1 pages 0,1
    bt_drop = torch.full_like(bt, -1)
    bt_drop[0, :3] = bt[0, [0, 2, 3]]
    bt_drop[1, :2] = bt[1, :2]
    np.testing.assert_allclose(got, oracle.decode(q, k, v, bt_drop, [12, 8], scale), rtol=0, atol=1e-12)


def test_context_clamped_to_table_row_and_empty_rows():
    q, k, v, bt, lens, scale = small_case(9, B=3, H=4, Hkv=1, D=8, bs=4, lens=[8, 5, 4])
    base = oracle.decode(q, k, v, bt, lens, scale)
    over = oracle.decode(q, k, v, bt, [8 + 100, 5, 4], scale)    # row holds 2 pages = 8 tokens
    np.testing.assert_array_equal(over[0], base[0])
    empty = oracle.decode(q, k, v, bt, [0, -3, 4], scale)
    assert np.all(empty[0] == 0) and np.all(empty[1] == 0)
    np.testing.assert_array_equal(empty[2], base[2])
    all_masked = oracle.decode(q, k, v, torch.full_like(bt, -1), lens, scale)
    assert np.all(all_masked == 0)


def test_poison_in_unreferenced_memory_does_not_leak():
    q, k, v, bt, lens, scale = small_case(10, B=2, H=4, Hkv=2, D=8, bs=4, lens=[6, 11], spare=3)
    base = oracle.decode(q, k, v, bt, lens, scale)
    kp, vp = k.clone(), v.clone()
    used = set(bt[bt >= 0].tolist())
    for blk in range(k.shape[0]):
        if blk not in used:
            kp[blk], vp[blk] = float("nan"), float("nan")
    kp[int(bt[0, 1]), 2:], vp[int(bt[0, 1]), 2:] = float("nan"), float("nan")   # slots past 6
    kp[int(bt[1, 2]), 3:], vp[int(bt[1, 2]), 3:] = 1e4, 1e4                     # slots past 11
    np.testing.assert_array_equal(oracle.decode(q, kp, vp, bt, lens, scale), base)


# --------------------------------------------------------------------------
# resolved page indices
# --------------------------------------------------------------------------
def test_resolve_blocks_hand_cases():
    bt = [[3, 1, -1, 0], [2, 9, 4, 1], [5, 6, 7, 8]]
    got = oracle.resolve_blocks(bt, [9, 16, 0], block_size=4, num_blocks=6)
    want = [[3, 1, -1, -1],      # 9 tokens -> pages 0..2; page 2 is -1
            [2, -1, 4, 1],       # 9 >= num_blocks -> masked
            [-1, -1, -1, -1]]    # empty sequence
    np.testing.assert_array_equal(got, want)


def test_resolve_blocks_bruteforce():
    g = np.random.default_rng(11)
    B, mb, bs, NB = 7, 9, 4, 20
    bt = g.integers(-3, NB + 3, size=(B, mb)).astype(np.int32)
    lens = g.integers(-2, mb * bs + 6, size=B).astype(np.int32)
    got = oracle.resolve_blocks(bt, lens, bs, NB)
    for b in range(B):
        pages_used = math.ceil(min(max(int(lens[b]), 0), mb * bs) / bs)
        for j in range(mb):
            e = int(bt[b, j])
            want = e if (j < pages_used and 0 <= e < NB) else -1
            assert got[b, j] == want, (b, j)


# --------------------------------------------------------------------------
# append of the new token
# --------------------------------------------------------------------------
def test_append_changes_exactly_the_addressed_slots():
    q, k, v, bt, lens, scale = small_case(12, B=4, H=8, Hkv=2, D=8, bs=4, lens=[5, 8, 1, 11], spare=3)
    g = torch.Generator().manual_seed(13)
    kn = torch.randn(4, 2, 8, generator=g).to(k.dtype)
    vn = torch.randn(4, 2, 8, generator=g).to(k.dtype)
    pos = torch.tensor([5, 7, -1, 400], dtype=torch.int32)   # seq 2 padding, seq 3 past its row
    k2, v2 = oracle.append_kv(k, v, kn, vn, bt, pos)
    changed = set()
    for b, p_ in enumerate(pos.tolist()):
        if 0 <= p_ < bt.shape[1] * 4 and int(bt[b, p_ // 4]) >= 0:
            e, s = int(bt[b, p_ // 4]), p_ % 4
            assert torch.equal(k2[e, s], kn[b]) and torch.equal(v2[e, s], vn[b])
            changed.add((e, s))
    mask = torch.ones(k.shape[:2], dtype=torch.bool)
    for e, s in changed:
        mask[e, s] = False
    assert torch.equal(k2[mask], k[mask]) and torch.equal(v2[mask], v[mask])
    assert len(changed) == 2


def test_append_skips_masked_entries():
    q, k, v, bt, lens, scale = small_case(14, B=2, H=4, Hkv=2, D=8, bs=4, lens=[6, 6], spare=2)
    bt = bt.clone()
    bt[0, 1] = -1
    bt[1, 1] = k.shape[0] + 3
    kn = torch.ones(2, 2, 8).to(k.dtype)
    k2, v2 = oracle.append_kv(k, v, kn, kn, bt, torch.tensor([5, 6], dtype=torch.int32))
    assert torch.equal(k2, k) and torch.equal(v2, v)


def test_append_then_decode_equals_decode_with_token_in_place():
    q, k, v, bt, lens, scale = small_case(15, B=3, H=8, Hkv=4, D=16, bs=4, lens=[6, 9, 12], spare=4)
    g = torch.Generator().manual_seed(16)
    kn = torch.randn(3, 4, 16, generator=g).to(k.dtype)
    vn = torch.randn(3, 4, 16, generator=g).to(k.dtype)
    pos = torch.tensor([6, 9, 11], dtype=torch.int32)       # last one overwrites an existing slot
    # cache with the token placed by hand, through an independent index computation
    kh, vh = k.clone(), v.clone()
    for b in range(3):
        p_ = int(pos[b])
        kh[int(bt[b, p_ // 4]), p_ % 4] = kn[b]
        vh[int(bt[b, p_ // 4]), p_ % 4] = vn[b]
    k2, v2 = oracle.append_kv(k, v, kn, vn, bt, pos)
    np.testing.assert_array_equal(oracle.decode(q, k2, v2, bt, pos + 1, scale),
                                  oracle.decode(q, kh, vh, bt, pos + 1, scale))


# --------------------------------------------------------------------------
# several query tokens per sequence (causal over the new tokens)
# --------------------------------------------------------------------------
def test_multi_token_rows_equal_one_token_decodes_of_their_prefix():
    B, Q, H, Hkv, D, bs = 3, 4, 8, 2, 16, 4
    _, k, v, bt, lens, scale = small_case(21, B=B, H=H, Hkv=Hkv, D=D, bs=bs, lens=[9, 14, 3])
    g = torch.Generator().manual_seed(22)
    q = torch.randn(B, Q, H, D, generator=g).to(k.dtype)
    got = oracle.decode_multi(q, k, v, bt, lens, scale)
    for i in range(Q):
        prefix = torch.clamp(lens - Q + i + 1, min=0)
        want = oracle.decode(q[:, i].contiguous(), k, v, bt, prefix, scale)
        np.testing.assert_array_equal(got[:, i], want)
    assert np.all(got[2, :1] == 0)          # T = 3 < Q: the first query sees no token


def test_multi_token_with_one_token_is_decode():
    q, k, v, bt, lens, scale = small_case(23, B=2, H=4, Hkv=4, D=8, bs=2, lens=[5, 7])
    np.testing.assert_array_equal(oracle.decode_multi(q[:, None], k, v, bt, lens, scale)[:, 0],
                                  oracle.decode(q, k, v, bt, lens, scale))


def test_multi_token_matches_causal_bruteforce():
    B, Q, H, Hkv, D, bs = 2, 3, 6, 3, 8, 4
    _, k, v, bt, lens, scale = small_case(24, B=B, H=H, Hkv=Hkv, D=D, bs=bs, lens=[10, 6])
    q = torch.randn(B, Q, H, D, generator=torch.Generator().manual_seed(25)).to(k.dtype)
    got = oracle.decode_multi(q, k, v, bt, lens, scale)
    kd, vd, qd = (t.to(torch.float64).numpy() for t in (k, v, q))
    sc = float(np.float32(scale))
    for b in range(B):
        T = int(lens[b])
        toks = np.arange(T)
        ent = bt.numpy()[b, toks // bs]
        Kb, Vb = kd[ent, toks % bs], vd[ent, toks % bs]       # [T, Hkv, D]
        for i in range(Q):
            mask = toks <= T - Q + i
            for h in range(H):
                s = sc * (Kb[:, h // (H // Hkv)] @ qd[b, i, h])
                s = np.where(mask, s, -np.inf)
                np.testing.assert_allclose(got[b, i, h], scipy.special.softmax(s) @ Vb[:, h // (H // Hkv)],
                                           rtol=0, atol=1e-12)


@pytest.mark.parametrize("threads", [1, 3, 7])
def test_threaded_driver_equals_decode(threads):
    """The multi-core baseline driver runs the same per-row arithmetic: its
    output is bit-identical to the single-threaded decode, whatever the split."""
    q, kc, vc, bt, lens, scale = small_case(41, B=3, H=8, Hkv=2, D=64, bs=16, lens=[0, 45, 130])
    want = oracle.decode(q, kc, vc, bt, lens, scale)
    got, used = oracle.decode_mt(q, kc, vc, bt, lens, scale, threads=threads)
    assert used == threads
    assert np.array_equal(got, want)


@pytest.mark.parametrize("threads", [1, 2, 5, 7, 20])
def test_threaded_multi_driver_equals_decode_multi(threads):
    """Pieces of (sequence, run of query tokens) through the multi-token oracle
    give its whole-batch result bit for bit, also with more threads than
    sequences (runs of query tokens shorter than Q, sequences shorter than Q)."""
    g = torch.Generator().manual_seed(43)
    q1, kc, vc, bt, lens, scale = small_case(43, B=5, H=8, Hkv=2, D=64, bs=16,
                                             lens=[3, 0, 45, 130, 17])
    q = torch.randn(5, 4, 8, 64, generator=g).to(torch.float16)
    want = oracle.decode_multi(q, kc, vc, bt, lens, scale)
    got, used = oracle.decode_multi_mt(q, kc, vc, bt, lens, scale, threads=threads)
    assert used == min(threads, 5 * 4)
    assert np.array_equal(got, want)
