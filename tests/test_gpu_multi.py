"""GPU parity of the multi-token step (q_len > 1, causal over the new tokens)
through the C ABI, against the fp64 oracle.

Bar: max |gpu - oracle| <= 2e-3 on fp32 output, as for the one-token decode.
Covered, on both kernels that serve several query tokens (the warp-level MMA
path with up to 16 rows per CTA, and the tcgen05 tile kernel with 128-row
tiles; the kernel switch forces one of them): every group size with q_len up to
and past 16 and 128 rows, sequences shorter than q_len (query tokens that see
nothing), masked table entries, every split mode (one pass, cluster,
workspace, balanced), the q-dtype output, the full-size multi-token
workloads whole, and the padding rows of Q tiles that persistent CTAs and the
balanced split load by TMA (another sequence's queries, poisoned with NaN).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_08_gb300 as pa
from paged_kv_attention_08_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = 2e-3
DEV = "cuda:0"


@pytest.fixture(params=["auto", "mma", "tile"])
def kernel(request, switches):
    """Which kernel serves the calls: the library's choice, or one forced."""
    switches(kernel=request.param)
    return request.param


def run(x, partition_tokens=0, out_dtype=torch.float32):
    """One call; the workspace is filled with NaN first, so that a read of a
    partial that no CTA wrote shows in the output."""
    out = torch.full(x.q.shape, float("nan"), dtype=out_dtype, device=x.q.device)
    need = pa.workspace_size_multi(x.q, x.k_cache, x.block_tables, out_dtype, x.max_context_len,
                                   partition_tokens)
    ws = torch.full((max(need, 16) // 4 + 1,), float("nan"), dtype=torch.float32, device=x.q.device)
    pa.decode_multi(out, x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens, x.scale,
                    x.max_context_len, partition_tokens, workspace=ws)
    torch.cuda.synchronize()
    return out


def check(got, want, tol=TOL):
    g = got.double().cpu().numpy()
    assert np.isfinite(g).all(), "non-finite output"
    err = np.abs(g - want).max()
    assert err <= tol, f"max abs err {err:.3e} > {tol}"


def multi_case(seed, B, Q, H, Hkv, D, bs, lens, dtype=torch.bfloat16, spare=3, mb_extra=1):
    g = torch.Generator().manual_seed(seed)
    pages = [(t + bs - 1) // bs for t in lens]
    mb = max(1, max(pages)) + mb_extra
    pool = sum(pages) + spare
    perm = torch.randperm(pool, generator=g)
    bt = torch.full((B, mb), -1, dtype=torch.int32)
    c = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[c:c + n].to(torch.int32)
        c += n
    spec = workloads.Spec("case", B, H, Hkv, D, bs, dtype, "list:" + ",".join(map(str, lens)),
                          q_len=Q)
    return workloads.Inputs(spec, torch.randn(B, Q, H, D, generator=g).to(dtype),
                            torch.randn(pool, bs, Hkv, D, generator=g).to(dtype),
                            torch.randn(pool, bs, Hkv, D, generator=g).to(dtype),
                            bt, torch.tensor(lens, dtype=torch.int32), 1.0 / math.sqrt(D),
                            max(lens), list(lens))


def oracle_of(x):
    return oracle.decode_multi(x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens, x.scale)


# (B, Q, H, Hkv, D, bs, lens): groups 1..16, Q below, at and past 16 / group
CASES = [
    (3, 2, 8, 8, 64, 16, [1, 37, 200]),       # G=1, 2 rows of 16
    (2, 16, 8, 8, 64, 32, [16, 333]),          # G=1, exactly 16 rows; T = Q
    (2, 17, 4, 4, 128, 16, [40, 129]),         # G=1, two chunks (16 + 1)
    (2, 3, 16, 8, 128, 16, [129, 7]),          # G=2
    (3, 4, 32, 8, 128, 16, [2, 64, 300]),      # G=4, 16 rows, one sequence shorter than Q
    (2, 5, 32, 8, 128, 32, [500, 31]),         # G=4, two chunks (4 + 1)
    (2, 2, 16, 2, 128, 16, [77, 1]),           # G=8
    (2, 3, 16, 1, 256, 32, [1000, 33]),        # G=16, three chunks of one token
    (2, 6, 8, 4, 256, 16, [100, 401]),         # G=2, 12 rows
    (2, 40, 16, 4, 128, 16, [45, 700]),        # G=4, 160 rows: two 128-row tiles
    (1, 130, 8, 8, 64, 32, [520]),             # G=1, 130 rows: a tile of 2 rows after 128
    (2, 24, 16, 1, 256, 32, [24, 1500]),       # G=16, 384 rows, a sequence exactly Q long
]
IDS = [f"B{c[0]}Q{c[1]}H{c[2]}kv{c[3]}D{c[4]}bs{c[5]}" for c in CASES]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_multi_token_vs_oracle(case, dtype, kernel):
    B, Q, H, Hkv, D, bs, lens = case
    x = multi_case(13, B, Q, H, Hkv, D, bs, lens, dtype)
    want = oracle_of(x)
    xd = x.to(DEV)
    pages = -(-max(lens) // bs)
    # one pass, automatic, two-page partitions (workspace), <= 8 partitions (cluster)
    for pt in [pages * bs, 0, 2 * bs, -(-pages // min(pages, 8)) * bs]:
        check(run(xd, pt), want)


@pytest.mark.parametrize("case", [CASES[0], CASES[3], CASES[4], CASES[6]], ids=lambda c: f"Q{c[1]}H{c[2]}kv{c[3]}")
def test_multi_token_balanced(case):
    """The balanced split keeps all of a unit's query tokens in one CTA."""
    B, Q, H, Hkv, D, bs, lens = case
    x = multi_case(17, B, Q, H, Hkv, D, bs, lens)
    want = oracle_of(x)
    xd = x.to(DEV)
    assert Q * (H // Hkv) <= 16
    for _ in range(2):
        check(run(xd, pa.PARTITION_BALANCED), want)


def test_multi_token_one_token_equals_decode():
    """q_len = 1 through the multi-token entry point is the one-token decode, bit for bit."""
    x = workloads.make("sweep_b4_t2048", seed=3, device=DEV)
    ref = torch.empty(x.q.shape, dtype=torch.float32, device=DEV)
    pa.decode_splitkv(ref, x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens, x.scale,
                      x.max_context_len, 0)
    got = torch.empty((x.q.shape[0], 1) + tuple(x.q.shape[1:]), dtype=torch.float32, device=DEV)
    pa.decode_multi(got, x.q[:, None].contiguous(), x.k_cache, x.v_cache, x.block_tables,
                    x.context_lens, x.scale, x.max_context_len, 0)
    torch.cuda.synchronize()
    assert torch.equal(got[:, 0], ref)


def test_multi_token_masking_and_qdtype_output(kernel):
    x = multi_case(19, 4, 4, 16, 4, 128, 16, [0, 3, 50, 90], torch.float16, mb_extra=0)
    NB = x.k_cache.shape[0]
    bt = x.block_tables.clone()
    bt[3, 1] = -1           # an unallocated page inside the context
    bt[2, 0] = NB + 3       # an id outside the pool
    x.block_tables = bt
    want = oracle_of(x)
    assert np.all(want[0] == 0) and np.all(want[1, 3] != 0) and np.all(want[1, 0] == 0)
    xd = x.to(DEV)
    for pt in [0, 16, 32]:
        check(run(xd, pt), want)
    got = run(xd, 0, out_dtype=torch.float16).double().cpu().numpy()
    want_r = torch.from_numpy(want).to(torch.float16).double().numpy()
    a = np.abs(want_r)
    ulp = np.where(a > 0, 2.0 ** (np.floor(np.log2(np.where(a > 0, a, 1.0))) - 10), 2.0 ** -24)
    assert (np.abs(got - want_r) <= TOL + ulp).all()


@pytest.mark.parametrize("name", ["tiny_q3", "tiny_q8"])
def test_tiny_multi_workloads(name, kernel):
    x = workloads.make(name, seed=0, device=DEV)
    want = oracle_of(x.to("cpu"))
    for pt in [0, 16, 64]:
        check(run(x, pt), want)


_WHOLE = {}


def whole_oracle(name, x):
    """The whole fp64 oracle output of a workload, on all host threads, computed
    once per workload (the kernel choices share it)."""
    if name not in _WHOLE:
        h = x.to("cpu")
        _WHOLE[name] = oracle.decode_multi_mt(h.q, h.k_cache, h.v_cache, h.block_tables,
                                              h.context_lens, h.scale)[0]
    return _WHOLE[name]


@pytest.mark.parametrize("name", ["spec_b16_t2048_q4", "spec_b4_t8192_q8", "chunk_b2_t4096_q64",
                                  "prefill_b16_t2048_q256"])
def test_multi_token_full_size_whole_output(name, kernel):
    """Full-size multi-token workloads, automatic split: every element of the
    output within 2e-3 of the whole fp64 oracle."""
    x = workloads.make(name, seed=0, device=DEV)
    got = run(x, 0)
    check(got, whole_oracle(name, x))


def test_tile_kernel_poison_and_permutation(switches):
    """Tile kernel: NaN in every unreferenced block and in the slots past each
    context leaves the output bit-identical; so does a permutation of the pool
    with the table remapped."""
    switches(kernel="tile")
    x = multi_case(23, 3, 20, 16, 2, 128, 16, [30, 250, 77], spare=6)
    xd = x.to(DEV)
    base = run(xd, 0)
    NB = x.k_cache.shape[0]
    used = set(x.block_tables[x.block_tables >= 0].tolist())
    k, v = xd.k_cache.clone(), xd.v_cache.clone()
    for blk in range(NB):
        if blk not in used:
            k[blk] = float("nan")
            v[blk] = float("nan")
    for b, t in enumerate(x.lens_host):
        last = int(x.block_tables[b, (t - 1) // 16])
        k[last, t % 16 or 16:] = float("nan")
        v[last, t % 16 or 16:] = float("nan")
    xp = workloads.Inputs(x.spec, xd.q, k, v, xd.block_tables, xd.context_lens, x.scale,
                          x.max_context_len, x.lens_host)
    assert torch.equal(run(xp, 0), base)
    perm = torch.randperm(NB, generator=torch.Generator().manual_seed(5))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(NB)
    bt = x.block_tables.clone()
    bt[bt >= 0] = inv[bt[bt >= 0].long()].to(torch.int32)
    xq = workloads.Inputs(x.spec, xd.q, xd.k_cache[perm.to(DEV)].contiguous(),
                          xd.v_cache[perm.to(DEV)].contiguous(), bt.to(DEV), xd.context_lens,
                          x.scale, x.max_context_len, x.lens_host)
    assert torch.equal(run(xq, 0), base)
    assert pa.device_error() == 0


@pytest.mark.parametrize("D,dt", [(64, torch.float16), (128, torch.bfloat16)],
                         ids=["d64_fp16", "d128_bf16"])
def test_tile_masked_v_rows_per_warpgroup(switches, D, dt):
    """Whole tiles up to head_dim 128 keep an O per softmax warpgroup, and each
    half of a block's keys goes to its P V MMAs once that half's warpgroup has
    written its P and zeroed the half's masked V rows (a V row read before it
    is zeroed puts 0 * NaN into O).  NaN in every slot past each context and in
    every unreferenced block, over 384 persistent units whose last blocks end
    at every 16-token offset: ten calls, each bit-identical to the unpoisoned
    result, which is exact against the oracle."""
    switches(kernel="auto")
    B = 24
    lens = [40 + 21 * b for b in range(B)]
    x = multi_case(47, B, 40, 32, 8, D, 16, lens, dtype=dt, spare=5)
    xd = x.to(DEV)
    plan = pa.plan_info(xd.q, xd.k_cache, xd.block_tables, xd.max_context_len, 0)
    assert plan["kernel"] == "tcgen05 tile" and plan["ctas"] < B * 8 * 2, plan
    base = run(xd, 0)
    check(base, oracle_of(x))
    NB = x.k_cache.shape[0]
    used = set(x.block_tables[x.block_tables >= 0].tolist())
    k, v = xd.k_cache.clone(), xd.v_cache.clone()
    for blk in range(NB):
        if blk not in used:
            k[blk] = float("nan")
            v[blk] = float("nan")
    for b, t in enumerate(x.lens_host):
        last = int(x.block_tables[b, (t - 1) // 16])
        k[last, t % 16 or 16:] = float("nan")
        v[last, t % 16 or 16:] = float("nan")
    xp = workloads.Inputs(x.spec, xd.q, k, v, xd.block_tables, xd.context_lens, x.scale,
                          x.max_context_len, x.lens_host)
    for _ in range(10):
        assert torch.equal(run(xp, 0), base)
    assert pa.device_error() == 0


def _slot(x, b, t):
    """(pool block, slot) of sequence b's token t."""
    bs = x.k_cache.shape[1]
    return int(x.block_tables[b, t // bs]), t % bs


def test_tile_fp16_p_edge_cases(switches):
    """fp16 inputs on the tile kernel, where P enters the P V MMA as one fp16
    part (11 significant bits): (a) a query token that sees one cached token
    returns that token's V exactly; (b) a token whose score exceeds every
    other by ~134 (natural log units) returns its V exactly (the other weights
    round to 0, the normaliser is 1); (c) weights in [1/2, 1], each V row +-1
    with the sign of its weight's fp16 rounding error so that the errors add
    up: the error against the oracle stays within one fp16 rounding per weight,
    2^-11 * max|V - O| <= 2^-10, and above 2^-14 (the case exercises the
    rounding), and the output is within 2e-5 of the same weights rounded once
    to fp16 with the normaliser summed from the rounded weights (unrounded
    weights differ from that by 1.7e-4 here, a bf16 part by 3.3e-4)."""
    switches(kernel="tile")
    dt = torch.float16
    G = 8
    # (a) T = Q: query token 0 sits at position 0 and sees token 0 alone
    x = multi_case(61, 2, 40, 16, 2, 128, 16, [40, 40], dtype=dt)
    got = run(x.to(DEV), 0).cpu()
    check(got, oracle_of(x))
    for b in range(2):
        for kvh in range(2):
            blk, sl = _slot(x, b, 0)
            v0 = x.v_cache[blk, sl, kvh].float()
            assert torch.equal(got[b, 0, kvh * G:(kvh + 1) * G], v0.expand(G, -1))
    # (b) one dominant token (token 0, seen by every query token)
    x = multi_case(62, 2, 40, 16, 2, 128, 16, [700, 300], dtype=dt)
    q = torch.zeros_like(x.q)
    q[..., 0] = 40.0
    k = x.k_cache.clone()
    k[..., 0] = k[..., 0].clamp(-2, 2)  # other scores <= 80 * scale
    for b in range(2):
        blk, sl = _slot(x, b, 0)
        k[blk, sl] = 0
        k[blk, sl, :, 0] = 40.0  # 1600 * scale
    xb = workloads.Inputs(x.spec, q, k, x.v_cache, x.block_tables, x.context_lens, x.scale,
                          x.max_context_len, x.lens_host)
    got = run(xb.to(DEV), 0).cpu()
    check(got, oracle_of(xb))
    for b in range(2):
        blk, sl = _slot(x, b, 0)
        for kvh in range(2):
            want = x.v_cache[blk, sl, kvh].float().expand(40, G, -1)
            assert torch.equal(got[b, :, kvh * G:(kvh + 1) * G], want)
    # (c) adversarial rounding: scores c_t (q = e_0, k_t = c_t e_0), the maximum
    # 8 at tokens 0 and 64 (both halves of the first block, so both softmax
    # warpgroups subtract the same maximum); the weight is computed here as the
    # kernel does, 2^fma(c_t, qscale, -8 qscale) in fp32, and V_t = sign of its
    # fp16 rounding error
    T = 1024
    x = multi_case(63, 1, 8, 8, 1, 128, 16, [T], dtype=dt)
    gen = torch.Generator().manual_seed(64)
    c = (torch.rand(T, generator=gen) * 7.8 + 0.2).to(dt)
    c[0] = 8.0
    c[64] = 8.0
    qscale = np.float32(np.float32(x.scale) * np.float32(1.4426950408889634))
    ms = np.float32(np.float32(8.0) * qscale)
    arg = (c.double().numpy() * float(qscale) - float(ms)).astype(np.float32).astype(np.float64)
    w = np.exp2(arg)
    sign = np.where(w.astype(np.float16).astype(np.float64) >= w, 1.0, -1.0)
    q = torch.zeros_like(x.q)
    q[..., 0] = 1.0
    k = torch.zeros_like(x.k_cache)
    v = torch.zeros_like(x.v_cache)
    for t in range(T):
        blk, sl = _slot(x, 0, t)
        k[blk, sl, 0, 0] = c[t]
        v[blk, sl, 0, :] = float(sign[t])
    xc = workloads.Inputs(x.spec, q, k, v, x.block_tables, x.context_lens, x.scale,
                          x.max_context_len, x.lens_host)
    xcd = xc.to(DEV)
    # one partition, so that both warpgroups subtract the maximum 8 qscale
    plan = pa.plan_info(xcd.q, xcd.k_cache, xcd.block_tables, xcd.max_context_len, T)
    assert plan["kernel"] == "tcgen05 tile" and plan["partitions"] == 1, plan
    got = run(xcd, T).double().cpu().numpy()  # [1, 8, 8, 128]
    err = np.abs(got - oracle_of(xc)).max()
    assert 2.0 ** -14 < err <= 2.0 ** -10, err
    p16 = w.astype(np.float16).astype(np.float64)
    for i in range(8):  # query token i sees tokens 0 .. T - 8 + i
        n = T - 8 + i + 1
        emu = (p16[:n] * sign[:n]).sum() / p16[:n].sum()
        assert np.abs(got[0, i] - emu).max() <= 2e-5, (i, np.abs(got[0, i] - emu).max())
    assert pa.device_error() == 0


def test_tile_output_16_byte_aligned(switches):
    """The tile kernel writes fp32 rows in whole 32-byte sectors when the output
    (or the workspace's partials) starts on a 32-byte boundary, else in 16-byte
    stores: an output and a workspace 16 bytes past a 32-byte boundary give
    results bit-identical to the aligned call, in one pass and through the
    workspace."""
    switches(kernel="tile")
    lens = [300, 77, 1000]
    x = multi_case(53, 3, 40, 16, 2, 128, 16, lens)
    xd = x.to(DEV)
    pages = -(-max(lens) // 16)
    n = xd.q.numel()

    def off16(numel):
        # a NaN-filled fp32 view of `numel` elements starting 16 bytes past a 32-byte boundary
        buf = torch.full((numel + 16,), float("nan"), dtype=torch.float32, device=DEV)
        k = (-(buf.data_ptr() // 4) % 8) + 4
        v = buf[k:k + numel]
        assert v.data_ptr() % 32 == 16
        return v

    for pt, reduce in [(pages * 16, "none"), (2 * 16, "workspace")]:
        plan = pa.plan_info(xd.q, xd.k_cache, xd.block_tables, xd.max_context_len, pt)
        assert plan["kernel"] == "tcgen05 tile" and reduce in plan["reduce"], plan
        want = run(xd, pt)
        need = pa.workspace_size_multi(xd.q, xd.k_cache, xd.block_tables, torch.float32,
                                       xd.max_context_len, pt)
        out = off16(n).view(xd.q.shape)
        ws = off16(max(need, 16) // 4 + 1)
        pa.decode_multi(out, xd.q, xd.k_cache, xd.v_cache, xd.block_tables, xd.context_lens,
                        xd.scale, xd.max_context_len, pt, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(out, want)
    assert pa.device_error() == 0


@pytest.mark.parametrize("Q,H,Hkv", [(1, 16, 1), (2, 16, 2)], ids=["mqa_q1", "g8_q2"])
def test_tile_compact_q_tile(switches, Q, H, Hkv):
    """Units of at most 16 rows at head_dim 256 stage a compact Q tile (the
    MMA's other rows read what follows it): exact against the oracle, bit-
    identical to whole 128-row Q tiles, and unchanged by NaN in every
    unreferenced block, in one pass and in cluster / workspace splits."""
    switches(kernel="auto")
    x = multi_case(29, 3, Q, H, Hkv, 256, 32, [70, 1000, 5], spare=6)
    want = oracle_of(x)
    xd = x.to(DEV)
    NB = x.k_cache.shape[0]
    used = set(x.block_tables[x.block_tables >= 0].tolist())
    k, v = xd.k_cache.clone(), xd.v_cache.clone()
    for blk in range(NB):
        if blk not in used:
            k[blk] = float("nan")
            v[blk] = float("nan")
    xp = workloads.Inputs(x.spec, xd.q, k, v, xd.block_tables, xd.context_lens, x.scale,
                          x.max_context_len, x.lens_host)
    for pt in [0, 32 * 32, 4 * 32]:
        switches(compact_q=1)
        compact = run(xd, pt)
        check(compact, want)
        assert torch.equal(run(xp, pt), compact)
        switches(compact_q=0)
        assert torch.equal(run(xd, pt), compact)
    assert pa.device_error() == 0


@pytest.mark.parametrize("case", ["whole_persistent", "whole_persistent_bf16", "whole_persistent_d64",
                                  "compact_persistent", "compact_balanced"])
def test_padding_rows_read_other_sequences_queries(switches, case):
    """A CTA's later segments (persistent CTAs, the balanced split) load their Q
    tile by TMA: the tile's rows past the unit's rows then hold the next query
    tokens, i.e. another sequence's queries (or the fill value past the last
    one), where a staged tile holds zeros.  Those rows are masked, so NaN
    queries in one sequence leave every other sequence's output exact.
    Cases: 40 tokens x 4 heads = 160 rows (a full and a partial 128-row tile)
    over 320 units, fp16 and bf16 at head_dim 128 and fp16 at 64; 3 tokens x
    4 heads = 12 rows at head_dim 256 (compact tiles) over 200 units; the same
    rows through the balanced split."""
    switches(kernel="auto")
    if case.startswith("whole_persistent"):
        D = 64 if case.endswith("d64") else 128
        dt = torch.bfloat16 if case.endswith("bf16") else torch.float16
        x = multi_case(41, 20, 40, 32, 8, D, 16, [40 + 7 * b for b in range(20)], dtype=dt)
        pt, units = 0, 20 * 8 * 2
    elif case == "compact_persistent":
        # (the automatic choice serves 12-row units with the warp-level kernel)
        switches(kernel="tile")
        x = multi_case(42, 200, 3, 4, 1, 256, 32, [3 + 5 * b for b in range(200)])
        pt, units = 0, 200
    else:
        x = multi_case(43, 24, 3, 8, 2, 256, 32, [3 + 37 * b for b in range(24)])
        pt, units = pa.PARTITION_BALANCED, 48
    want = oracle_of(x)
    poisoned = 5
    q = x.q.clone()
    q[poisoned] = float("nan")
    xn = workloads.Inputs(x.spec, q, x.k_cache, x.v_cache, x.block_tables, x.context_lens,
                          x.scale, x.max_context_len, x.lens_host)
    xd = xn.to(DEV)
    plan = pa.plan_info(xd.q, xd.k_cache, xd.block_tables, xd.max_context_len, pt)
    assert plan["kernel"] == "tcgen05 tile", plan
    if pt == pa.PARTITION_BALANCED:
        assert plan["reduce"] == "balanced split", plan
    else:
        assert plan["partitions"] == 1 and plan["ctas"] < units, plan  # persistent CTAs
    got = run(xd, pt)
    keep = [b for b in range(x.q.shape[0]) if b != poisoned]
    check(got[keep], want[keep])
    assert pa.device_error() == 0
