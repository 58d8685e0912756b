"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bar: max |gpu - oracle| <= 2e-3 on fp32 output (fp16/bf16 K/V, fp32
accumulate); q-dtype output within 2e-3 plus one ulp of the oracle rounded to
that dtype; bit-exact page indices; bit-identical output under pool
permutation and poison in unreferenced memory.
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


def run(x, mode="single", out_dtype=torch.float32, partition_tokens=0):
    out = torch.full(x.q.shape, float("nan"), dtype=out_dtype, device=x.q.device)
    if mode == "single":
        pa.decode(out, x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens, x.scale)
    else:
        # a NaN-filled workspace: a read of a partial that no CTA wrote shows
        need = pa.workspace_size(x.q, x.k_cache, x.block_tables, out_dtype, x.max_context_len,
                                 partition_tokens)
        ws = torch.full((max(need, 16) // 4 + 1,), float("nan"), dtype=torch.float32,
                        device=x.q.device)
        pa.decode_splitkv(out, x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens, x.scale,
                          x.max_context_len, partition_tokens, workspace=ws)
    torch.cuda.synchronize()
    return out


def assert_close_fp32(got, want, tol=TOL):
    g = got.double().cpu().numpy()
    assert np.isfinite(g).all(), "non-finite output"
    err = np.abs(g - want).max()
    assert err <= tol, f"max abs err {err:.3e} > {tol}"
    return err


# ---------------------------------------------------------------------------
# workloads small enough for the whole oracle
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["tiny", "sweep_b1_t512", "sweep_b16_t256", "sweep_b4_t2048",
                                  "tiny_mqa"])
@pytest.mark.parametrize("mode,pages", [("single", 0), ("split", 0), ("split", 1), ("split", 4)])
def test_small_workloads_vs_oracle(name, mode, pages):
    """Whole oracle; explicit partitions of one and of four pages."""
    x = workloads.make(name, seed=0, device=DEV)
    want = oracle.decode(x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens, x.scale)
    pt = pages * x.k_cache.shape[1]
    assert_close_fp32(run(x, mode, partition_tokens=pt), want)


@pytest.mark.parametrize("name", ["tiny", "sweep_b4_t2048"])
@pytest.mark.parametrize("mode", ["single", "split"])
def test_qdtype_output(name, mode):
    x = workloads.make(name, seed=1, device=DEV)
    want = oracle.decode(x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens, x.scale)
    got = run(x, mode, out_dtype=x.q.dtype).double().cpu().numpy()
    want_r = torch.from_numpy(want).to(x.q.dtype).double().numpy()   # RNE to the output dtype
    mant = 7 if x.q.dtype == torch.bfloat16 else 10
    a = np.abs(want_r)
    ulp = np.where(a > 0, 2.0 ** (np.floor(np.log2(np.where(a > 0, a, 1.0))) - mant), 2.0 ** -24)
    assert np.isfinite(got).all()
    assert (np.abs(got - want_r) <= TOL + ulp).all()


# ---------------------------------------------------------------------------
# full-size workloads: every output element against the whole oracle (run on
# all host threads, computed once per workload)
# ---------------------------------------------------------------------------
_WHOLE = {}


def whole_oracle(name, x):
    if name not in _WHOLE:
        h = x.to("cpu")
        _WHOLE[name] = oracle.decode_mt(h.q, h.k_cache, h.v_cache, h.block_tables,
                                        h.context_lens, h.scale)[0]
    return _WHOLE[name]


@pytest.mark.parametrize("name,mode,pt", [
    ("ragged_b64", "single", 0), ("ragged_b64", "split", 0), ("ragged_b64", "split", 512),
    ("long_b1_t8192", "split", 512), ("long_b1_t32768", "split", 512),
    ("long_b1_t131072", "split", 512), ("long_b4_t8192", "split", 512),
    ("long_b4_t32768", "split", 512), ("long_b4_t131072", "split", 512),
    ("long_b1_t8192", "split", 0), ("long_b1_t32768", "split", 0),
    ("long_b1_t131072", "split", 0), ("long_b4_t8192", "split", 0),
    ("long_b4_t32768", "split", 0), ("long_b4_t131072", "split", 0),
    ("long_b4_t32768", "single", 0),
    ("mqa_b32_t16384", "split", 0), ("mqa_b32_t16384", "single", 0),
])
def test_full_size_whole_output(name, mode, pt):
    """The five configurations' full-size workloads, in the launch
    configuration the bench times (automatic split) and with the long group's
    own 512-token partitions: every element within 2e-3 of the fp64 oracle."""
    x = workloads.make(name, seed=0, device=DEV)
    got = run(x, mode, partition_tokens=pt)
    assert_close_fp32(got, whole_oracle(name, x))


# ---------------------------------------------------------------------------
# other instantiations: head_dim 64/256, groups 1/2/8/16, block 16/32
# ---------------------------------------------------------------------------
def random_case(seed, B, H, Hkv, D, bs, lens, dtype, spare=5, mb_extra=1):
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
    spec = workloads.Spec("case", B, H, Hkv, D, bs, dtype, "list:" + ",".join(map(str, lens)))
    x = workloads.Inputs(spec, torch.randn(B, H, D, generator=g).to(dtype),
                         torch.randn(pool, bs, Hkv, D, generator=g).to(dtype),
                         torch.randn(pool, bs, Hkv, D, generator=g).to(dtype),
                         bt, torch.tensor(lens, dtype=torch.int32), 1.0 / math.sqrt(D),
                         max(lens), list(lens))
    return x


SHAPES = [
    dict(B=3, H=8, Hkv=8, D=64, bs=16, lens=[1, 37, 200]),
    dict(B=2, H=8, Hkv=4, D=64, bs=32, lens=[64, 333]),
    dict(B=2, H=16, Hkv=2, D=128, bs=16, lens=[129, 7]),
    dict(B=2, H=32, Hkv=8, D=128, bs=32, lens=[500, 31]),
    dict(B=2, H=16, Hkv=1, D=256, bs=32, lens=[1000, 33]),
    dict(B=3, H=4, Hkv=4, D=256, bs=16, lens=[17, 256, 2]),
    dict(B=2, H=8, Hkv=4, D=256, bs=16, lens=[100, 401]),
    dict(B=1, H=16, Hkv=2, D=64, bs=16, lens=[777]),
]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"H{s['H']}kv{s['Hkv']}D{s['D']}bs{s['bs']}")
def test_other_shapes(shape, dtype):
    x = random_case(3, dtype=dtype, **shape)
    want = oracle.decode(x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens, x.scale)
    xd = x.to(DEV)
    for mode, pt in [("single", 0), ("split", 0), ("split", shape["bs"] * 2)]:
        assert_close_fp32(run(xd, mode, partition_tokens=pt), want)


@pytest.mark.parametrize("parts", [2, 3, 5, 8])
@pytest.mark.parametrize("shape", [SHAPES[2], SHAPES[3], SHAPES[4], SHAPES[0]],
                         ids=lambda s: f"H{s['H']}kv{s['Hkv']}D{s['D']}bs{s['bs']}")
def test_cluster_split_sizes(shape, parts):
    """Splits of at most 8 partitions reduce inside one thread-block cluster."""
    x = random_case(7, dtype=torch.bfloat16, **shape)
    bs = shape["bs"]
    pages = -(-max(shape["lens"]) // bs)
    if pages < parts:
        pytest.skip("fewer pages than partitions")
    pt = -(-pages // parts) * bs
    assert -(-max(shape["lens"]) // pt) <= 8
    want = oracle.decode(x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens, x.scale)
    xd = x.to(DEV)
    ws = pa.workspace_size(xd.q, xd.k_cache, xd.block_tables, torch.float32, xd.max_context_len, pt)
    units = shape["B"] * shape["Hkv"]
    if units <= 8:
        assert ws == 0      # a handful of clusters always fits: reduced in the cluster
    # (16 clusters of 8 CTAs do not all fit at once on a 152-SM part: the
    # partitions then go through the workspace, which workspace_size reports)
    assert_close_fp32(run(xd, "split", partition_tokens=pt), want)


BALANCED_CASES = [
    dict(B=9, H=8, Hkv=2, D=128, bs=16, lens=[300, 0, 17, 1, 2000, 64, 0, 999, 15]),
    dict(B=3, H=16, Hkv=1, D=256, bs=32, lens=[5000, 31, 2900]),
    dict(B=5, H=8, Hkv=8, D=64, bs=16, lens=[1, 2, 3, 4, 5]),
    dict(B=1, H=32, Hkv=8, D=128, bs=32, lens=[7777]),
    dict(B=4, H=16, Hkv=2, D=64, bs=32, lens=[0, 0, 0, 0]),
    # fewer pages than CTAs: empty shares lie between a unit's CTAs
    dict(B=2, H=16, Hkv=8, D=128, bs=16, lens=[129, 7]),
    dict(B=2, H=16, Hkv=2, D=128, bs=16, lens=[77, 1]),
    dict(B=3, H=8, Hkv=8, D=64, bs=16, lens=[1, 37, 200]),
]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("case", BALANCED_CASES, ids=lambda s: f"B{s['B']}H{s['H']}kv{s['Hkv']}D{s['D']}")
def test_balanced_split(case, dtype):
    """The balanced split: equal shares of all pages per SM, straddling pieces
    combined afterwards (empty sequences, one-page units, units spread over
    many CTAs, CTAs holding several whole units)."""
    x = random_case(11, dtype=dtype, **case)
    want = oracle.decode(x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens, x.scale)
    xd = x.to(DEV)
    assert pa.workspace_size(xd.q, xd.k_cache, xd.block_tables, torch.float32,
                             xd.max_context_len, pa.PARTITION_BALANCED) > 0
    for _ in range(2):      # the second call reuses the workspace records
        assert_close_fp32(run(xd, "split", partition_tokens=pa.PARTITION_BALANCED), want)


# ---------------------------------------------------------------------------
# edge cases and invariances
# ---------------------------------------------------------------------------
def test_edge_lengths_and_masking():
    x = random_case(5, B=6, H=8, Hkv=2, D=128, bs=16, lens=[0, 1, 15, 16, 17, 95], dtype=torch.bfloat16,
                    mb_extra=0)
    NB = x.k_cache.shape[0]
    bt = x.block_tables.clone()
    bt[5, 2] = -1            # unallocated entry inside the context
    bt[4, 1] = NB + 7        # id outside the pool
    x.block_tables = bt
    lens = torch.tensor([0, 1, 15, 16, 17, 10_000], dtype=torch.int32)   # last: clamped to the row
    x.context_lens = lens
    x.lens_host = lens.tolist()
    want = oracle.decode(x.q, x.k_cache, x.v_cache, bt, lens, x.scale)
    xd = x.to(DEV)
    xd.max_context_len = 10_000
    for mode, pt in [("single", 0), ("split", 16), ("split", 32), ("split", 48), ("split", 0)]:
        got = run(xd, mode, partition_tokens=pt)
        assert_close_fp32(got, want)
        assert torch.all(got[0] == 0)        # empty context -> zeros


def test_all_masked_and_empty_batch():
    x = random_case(6, B=2, H=4, Hkv=4, D=128, bs=16, lens=[40, 20], dtype=torch.float16)
    x.block_tables = torch.full_like(x.block_tables, -1)
    xd = x.to(DEV)
    for mode, pt in [("single", 0), ("split", 16), ("split", 0)]:
        assert torch.all(run(xd, mode, partition_tokens=pt) == 0)
    e = workloads.make("tiny", device=DEV)
    out = torch.empty(0, 32, 128, device=DEV)
    pa.decode(out, e.q[:0], e.k_cache, e.v_cache, e.block_tables[:0], e.context_lens[:0], e.scale)


@pytest.mark.parametrize("mode,pt", [("single", 0), ("split", 32)])
def test_poison_does_not_leak(mode, pt):
    x = workloads.make("sweep_b16_t256", seed=2, device=DEV)
    lens = torch.randint(1, 257, (16,), generator=torch.Generator().manual_seed(3)).to(torch.int32)
    x.context_lens = lens.to(DEV)
    clean = run(x, mode, partition_tokens=pt)
    k, v = x.k_cache.clone(), x.v_cache.clone()
    bt = x.block_tables.cpu()
    for b in range(16):
        t = int(lens[b])
        last = int(bt[b, (t - 1) // 16])
        k[last, (t - 1) % 16 + 1:] = float("nan")
        v[last, (t - 1) % 16 + 1:] = float("nan")
        for j in range((t + 15) // 16, bt.shape[1]):        # pages past the context
            k[int(bt[b, j])] = float("nan")
            v[int(bt[b, j])] = float("nan")
    x.k_cache, x.v_cache = k, v
    poisoned = run(x, mode, partition_tokens=pt)
    assert torch.equal(poisoned, clean)


@pytest.mark.parametrize("mode,pt", [("single", 0), ("split", 64)])
def test_pool_permutation_bit_identical(mode, pt):
    x = workloads.make("ragged_b64", seed=4, device=DEV)
    base = run(x, mode, partition_tokens=pt)
    NB = x.k_cache.shape[0]
    perm = torch.randperm(NB, generator=torch.Generator().manual_seed(9)).to(DEV)
    k2, v2 = torch.empty_like(x.k_cache), torch.empty_like(x.v_cache)
    k2[perm], v2[perm] = x.k_cache, x.v_cache
    bt = x.block_tables
    x.block_tables = torch.where(bt >= 0, perm[bt.clamp(min=0).long()].to(torch.int32), bt)
    x.k_cache, x.v_cache = k2, v2
    assert torch.equal(run(x, mode, partition_tokens=pt), base)


def test_workspace_takes_any_contents_and_serves_shapes_in_turn():
    """Workspace splits need no clearing of the workspace: one workspace serves
    calls of different shapes in turn (each call's partials land where another
    call's were), workspaces of zeros, 0xFF bytes or random bytes, and graph
    replays of one captured call with the output poisoned in between all give
    the oracle's result."""
    cases = [("long_b1_t32768", 1728), ("ragged_b64", 256), ("long_b1_t8192", 432),
             ("sweep_b4_t2048", 128)]
    xs = [(workloads.make(n, seed=6, device=DEV), pt) for n, pt in cases]
    wants = []
    for x, pt in xs:
        info = pa.plan_info(x.q, x.k_cache, x.block_tables, x.max_context_len, pt)
        assert info["reduce"] == "workspace+combine kernel", info
        h = x.to("cpu")
        wants.append(oracle.decode_mt(h.q, h.k_cache, h.v_cache, h.block_tables,
                                      h.context_lens, h.scale)[0])
    need = max(pa.workspace_size(x.q, x.k_cache, x.block_tables, torch.float32,
                                 x.max_context_len, pt) for x, pt in xs)
    g = torch.Generator(device=DEV).manual_seed(3)
    fills = [torch.zeros(need, dtype=torch.uint8, device=DEV),
             torch.full((need,), 0xFF, dtype=torch.uint8, device=DEV),
             torch.randint(0, 256, (need,), generator=g, device=DEV).to(torch.uint8)]
    for ws in fills:
        for _ in range(2):                       # shapes in turn on one workspace
            for (x, pt), want in zip(xs, wants):
                out = torch.full(x.q.shape, float("nan"), dtype=torch.float32, device=DEV)
                pa.decode_splitkv(out, x.q, x.k_cache, x.v_cache, x.block_tables,
                                  x.context_lens, x.scale, x.max_context_len, pt, workspace=ws)
                torch.cuda.synchronize()
                assert_close_fp32(out, want)
    # graph replays of one captured call, the partials poisoned in between
    x, pt = xs[0]
    ws = fills[2]
    out = torch.full(x.q.shape, float("nan"), dtype=torch.float32, device=DEV)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        pa.decode_splitkv(out, x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens,
                          x.scale, x.max_context_len, pt, workspace=ws, stream=st)
        st.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=st):
            pa.decode_splitkv(out, x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens,
                              x.scale, x.max_context_len, pt, workspace=ws,
                              stream=torch.cuda.current_stream())
    for _ in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert_close_fp32(out, wants[0])
    assert pa.device_error() == 0


def test_split_count_invariance():
    x = workloads.make("long_b1_t32768", seed=5, device=DEV)
    host = x.to("cpu")
    want = oracle.decode_mt(host.q, host.k_cache, host.v_cache, host.block_tables,
                            host.context_lens, host.scale)[0]
    outs = []
    for mode, pt in [("single", 0), ("split", 16), ("split", 256), ("split", 512), ("split", 4096),
                     ("split", 0), ("split", pa.PARTITION_BALANCED)]:
        got = run(x, mode, partition_tokens=pt)
        assert_close_fp32(got, want)
        outs.append(got)
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= 1e-5


@pytest.mark.parametrize("name", ["tiny", "ragged_b64", "mqa_b32_t16384"])
def test_resolve_blocks_bit_exact(name):
    x = workloads.make(name, seed=0, device=DEV)
    got = torch.empty_like(x.block_tables)
    pa.resolve_blocks(got, x.block_tables, x.context_lens, x.k_cache.shape[1], x.k_cache.shape[0])
    torch.cuda.synchronize()
    want = oracle.resolve_blocks(x.block_tables, x.context_lens, x.k_cache.shape[1], x.k_cache.shape[0])
    np.testing.assert_array_equal(got.cpu().numpy(), want)


def test_resolve_blocks_garbage_tables():
    g = np.random.default_rng(12)
    B, mb, bs, NB = 33, 17, 16, 50
    bt = torch.from_numpy(g.integers(-5, NB + 5, size=(B, mb)).astype(np.int32))
    lens = torch.from_numpy(g.integers(-3, mb * bs + 40, size=B).astype(np.int32))
    got = torch.empty(B, mb, dtype=torch.int32, device=DEV)
    pa.resolve_blocks(got, bt.to(DEV), lens.to(DEV), bs, NB)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got.cpu().numpy(), oracle.resolve_blocks(bt, lens, bs, NB))


def test_workspace_errors_and_no_device_error():
    x = workloads.make("long_b1_t8192", device=DEV)
    out = torch.empty(x.q.shape, dtype=torch.float32, device=DEV)
    need = pa.workspace_size(x.q, x.k_cache, x.block_tables, torch.float32, x.max_context_len, 512)
    assert need > 0
    small = torch.empty(need - 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(pa.PaError) as ei:
        pa.decode_splitkv(out, x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens, x.scale,
                          x.max_context_len, 512, workspace=small)
    assert ei.value.code == 3
    with pytest.raises(pa.PaError):
        pa.decode_splitkv(out, x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens, x.scale,
                          x.max_context_len, 100)        # not a multiple of block_size
    assert pa.device_error() == 0


def test_bounded_wait_reports_timeout_and_context_survives():
    """A wait that can never complete gives up after its limit, the error word
    says PA_ERR_TIMEOUT, and the context keeps working."""
    assert pa.device_error() == 0
    pa.selftest_wait_timeout(20_000_000)      # 20 ms
    assert pa.device_error() == 5              # PA_ERR_TIMEOUT, and the word is cleared
    assert pa.device_error() == 0
    x = workloads.make("tiny", seed=0, device=DEV)
    want = oracle.decode(x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens, x.scale)
    assert_close_fp32(run(x, "split", partition_tokens=16), want)
    assert pa.device_error() == 0


# ---------------------------------------------------------------------------
# append of the new token
# ---------------------------------------------------------------------------
def _as_bits(t):
    return t.contiguous().view(torch.int16).cpu()


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("shape", [SHAPES[2], SHAPES[4], SHAPES[0]],
                         ids=lambda s: f"H{s['H']}kv{s['Hkv']}D{s['D']}bs{s['bs']}")
def test_append_bit_exact(shape, dtype):
    x = random_case(8, dtype=dtype, **shape)
    B, Hkv, D, bs = shape["B"], shape["Hkv"], shape["D"], shape["bs"]
    g = torch.Generator().manual_seed(9)
    kn = torch.randn(B, Hkv, D, generator=g).to(dtype)
    vn = torch.randn(B, Hkv, D, generator=g).to(dtype)
    mb = x.block_tables.shape[1]
    pos = torch.tensor([(7 * b + 3) % (mb * bs) for b in range(B)], dtype=torch.int32)
    pos[0] = -1                                    # padding sequence
    bt = x.block_tables.clone()
    if B > 2:
        bt[2, :] = -1                              # masked entry
    k_want, v_want = oracle.append_kv(x.k_cache, x.v_cache, kn, vn, bt, pos)
    kd, vd = x.k_cache.to(DEV), x.v_cache.to(DEV)
    pa.append_kv(kd, vd, kn.to(DEV), vn.to(DEV), bt.to(DEV), pos.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(_as_bits(kd), _as_bits(k_want))
    assert torch.equal(_as_bits(vd), _as_bits(v_want))


def test_append_then_decode_in_a_graph():
    """A decode iteration: append the new token (the last of each context),
    then attend; captured once in a CUDA graph and replayed."""
    x = workloads.make("ragged_b64", seed=3, device=DEV)
    host = x.to("cpu")                                   # the cache before any append
    B, _, D = x.q.shape
    Hkv = x.k_cache.shape[2]
    g = torch.Generator(device=DEV).manual_seed(4)
    kn = torch.randn(B, Hkv, D, generator=g, device=DEV).to(x.q.dtype)
    vn = torch.randn(B, Hkv, D, generator=g, device=DEV).to(x.q.dtype)
    pos = (x.context_lens - 1).contiguous()
    out = torch.empty(x.q.shape, dtype=torch.float32, device=DEV)
    need = pa.workspace_size(x.q, x.k_cache, x.block_tables, torch.float32, x.max_context_len, 0)
    ws = torch.empty(max(16, need), dtype=torch.uint8, device=DEV)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        def step():
            pa.append_kv(x.k_cache, x.v_cache, kn, vn, x.block_tables, pos, stream=st)
            pa.decode_splitkv(out, x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens,
                              x.scale, x.max_context_len, 0, workspace=ws, stream=st)
        step()
        st.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=st):
            step()
        out.fill_(float("nan"))
        graph.replay()
        st.synchronize()
    k2, v2 = oracle.append_kv(host.k_cache, host.v_cache, kn.cpu(), vn.cpu(), host.block_tables,
                              pos.cpu())
    assert torch.equal(_as_bits(x.k_cache), _as_bits(k2))
    want = oracle.decode_mt(host.q, k2, v2, host.block_tables, host.context_lens, host.scale)[0]
    assert_close_fp32(out, want)


@pytest.mark.parametrize("B,T,Hkv", [(2, 2048, 8), (4, 1024, 4), (16, 1500, 1)])
def test_sixteen_unit_automatic_plan(B, T, Hkv):
    """16 (sequence, kv head) units: the automatic plan sizes its clusters so
    that all of them are resident at once; exact against the oracle."""
    H = Hkv * 4
    spec = workloads.Spec("u16", B, H, Hkv, 128, 16, torch.bfloat16, f"fixed:{T}")
    x = workloads.make(spec, seed=9, device="cpu")
    want = oracle.decode(x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens, x.scale)
    xd = x.to(DEV)
    assert_close_fp32(run(xd, "split", partition_tokens=0), want)


# units (sequences x kv heads) around the number of clusters of 8 / 4 / 2 CTAs
# the device holds at once, and around 152 CTAs (the change of CTA shape)
EXACT_WS = [(8, u) for u in (8, 15, 16, 19, 20)] + [(4, u) for u in (32, 36, 37, 38, 40)] + \
           [(2, u) for u in (64, 76, 77, 80)]


@pytest.mark.parametrize("parts,units", EXACT_WS, ids=lambda v: str(v))
@pytest.mark.parametrize("kernel", ["auto", "tile"])
def test_workspace_size_is_exact_for_explicit_splits(parts, units, kernel, switches):
    """An explicit partition count: a workspace of exactly the reported size
    (none when it is 0) serves the call, whose reduction is the one plan_info
    reports; exact against the oracle."""
    switches(kernel=kernel)
    T = parts * 4 * 16
    x = random_case(31, B=units, H=4, Hkv=1, D=128, bs=16, lens=[T] * units,
                    dtype=torch.float16, spare=0, mb_extra=0)
    want = oracle.decode(x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens, x.scale)
    xd = x.to(DEV)
    pt = 4 * 16
    need = pa.workspace_size(xd.q, xd.k_cache, xd.block_tables, torch.float32, T, pt)
    info = pa.plan_info(xd.q, xd.k_cache, xd.block_tables, T, pt)
    assert info["partitions"] == parts
    assert (need > 0) == (info["reduce"] == "workspace+combine kernel"), (need, info)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=DEV)
    out = torch.full(xd.q.shape, float("nan"), dtype=torch.float32, device=DEV)
    pa.decode_splitkv(out, xd.q, xd.k_cache, xd.v_cache, xd.block_tables, xd.context_lens,
                      xd.scale, T, pt, workspace=ws)
    torch.cuda.synchronize()
    assert_close_fp32(out, want)
