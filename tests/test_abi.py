"""CPU-side checks of the C ABI: the library loads, exports every entry point
that include/*.h declares, and its host logic (status strings, validation,
partition choice, workspace sizing) behaves as documented.  No call here
reaches a kernel launch: every decode call is built to fail validation first.
"""
import ctypes
import glob
import os
import re

import numpy as np
import pytest
import torch

import paged_kv_attention_08_gb300 as pa
from paged_kv_attention_08_gb300 import build as pa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_entry_points():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    pa_build.build()
    pa._load()
    return pa._lib


def test_library_exports_every_declared_symbol(lib):
    names = declared_entry_points()
    assert {"pa_decode", "pa_decode_splitkv", "pa_workspace_size", "pa_resolve_blocks",
            "pa_status_string", "pa_choose_partition_tokens", "pa_device_error",
            "pa_selftest_wait_timeout", "pa_decode_splitkv_noalloc", "pa_decode_multi",
            "pa_workspace_size_multi"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings(lib):
    for code in range(6):
        assert lib.pa_status_string(code)
    assert lib.pa_status_string(99) == b"unknown status"


def shape(**kw):
    base = dict(batch=4, num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                max_blocks_per_seq=128, num_blocks=512, kv_dtype=pa.F16, out_dtype=pa.F32)
    base.update(kw)
    return pa._Shape(**base)


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails before any launch


@pytest.mark.parametrize("kw,code", [
    (dict(num_heads=30), 1),                 # H % Hkv != 0
    (dict(batch=-1), 1),
    (dict(max_blocks_per_seq=0), 1),
    (dict(num_blocks=0), 1),
    (dict(head_dim=96), 2),
    (dict(block_size=8), 2),
    (dict(num_heads=24, num_kv_heads=8), 2),  # group 3
    (dict(kv_dtype=pa.F32), 2),
    (dict(out_dtype=pa.BF16), 2),             # neither fp32 nor the kv dtype
    (dict(num_blocks=1 << 31), 2),
])
def test_shape_validation(lib, kw, code):
    s = shape(**kw)
    rc = lib.pa_decode(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), 0.1, None)
    assert rc == code
    rc = lib.pa_decode_splitkv(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), 0.1, 100, 0,
                               FAKE, 1 << 20, None)
    assert rc == code


def test_pointer_validation(lib):
    s = shape()
    assert lib.pa_decode(None, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), 0.1, None) == 1
    assert lib.pa_decode(FAKE + 8, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), 0.1, None) == 1
    assert lib.pa_decode(FAKE, FAKE, FAKE, FAKE, FAKE + 2, FAKE, ctypes.byref(s), 0.1, None) == 1
    assert lib.pa_decode(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0.1, None) == 1
    # split-only arguments
    assert lib.pa_decode_splitkv(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), 0.1, -1, 0,
                                 FAKE, 1 << 20, None) == 1
    assert lib.pa_decode_splitkv(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), 0.1, 100, 24,
                                 FAKE, 1 << 20, None) == 1
    assert lib.pa_decode_splitkv(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), 0.1, 100, -2,
                                 FAKE, 1 << 20, None) == 1
    # an empty batch is a no-op, whatever the pointers
    e = shape(batch=0)
    assert lib.pa_decode(None, None, None, None, None, None, ctypes.byref(e), 0.1, None) == 0
    assert lib.pa_resolve_blocks(None, FAKE, FAKE, ctypes.byref(s), None) == 1


@pytest.mark.parametrize("scale", [0.0, -0.1, float("inf"), float("nan")])
def test_scale_must_be_positive_and_finite(lib, scale):
    s = shape()
    assert lib.pa_decode(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), scale, None) == 1
    assert lib.pa_decode_splitkv(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), scale, 100, 0,
                                 FAKE, 1 << 20, None) == 1
    assert lib.pa_decode_multi(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), 2, scale, 100,
                               0, FAKE, 1 << 20, None) == 1
    assert lib.pa_decode_splitkv_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), scale,
                                         100, 0, None) == 1


def test_multi_token_validation(lib):
    s = shape()
    for q_len in (0, -3):
        assert lib.pa_decode_multi(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), q_len, 0.1,
                                   100, 0, FAKE, 1 << 20, None) == 1
        assert lib.pa_workspace_size_multi(ctypes.byref(s), q_len, 100, 16) == 0
    bad = shape(head_dim=96)
    assert lib.pa_decode_multi(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(bad), 2, 0.1, 100,
                               0, FAKE, 1 << 20, None) == 2
    e = shape(batch=0)
    assert lib.pa_decode_multi(None, None, None, None, None, None, ctypes.byref(e), 4, 0.1, 0, 0,
                               None, 0, None) == 0


def test_multi_token_workspace_size(lib):
    # B=4, H=32 (G=4), q_len 6: rows per partition B*H*Q; 131072 tokens in 256 partitions of 512
    s = shape(batch=4, max_blocks_per_seq=8192)
    rows = 4 * 32 * 6 * 256
    acc = rows * 128 * 4
    want = (acc + 255) // 256 * 256 + rows * 2 * 4
    assert lib.pa_workspace_size_multi(ctypes.byref(s), 6, 131072, 512) == want
    assert lib.pa_workspace_size_multi(ctypes.byref(s), 1, 131072, 512) == \
        lib.pa_workspace_size(ctypes.byref(s), 131072, 512)
    assert lib.pa_workspace_size_multi(ctypes.byref(s), 6, 131072, 131072) == 0   # one partition
    # up to 16 rows (q_len 4 x group 4) run on the warp-level MMA path, more on
    # the tile kernel; on both, <= 8 partitions reduce in a cluster, more go
    # through the workspace
    assert lib.pa_workspace_size_multi(ctypes.byref(s), 4, 8 * 512, 512) == 0
    assert lib.pa_workspace_size_multi(ctypes.byref(s), 6, 8 * 512, 512) == 0
    rows = 4 * 32 * 6 * 9
    assert lib.pa_workspace_size_multi(ctypes.byref(s), 6, 9 * 512, 512) == \
        (rows * 128 * 4 + 255) // 256 * 256 + rows * 2 * 4


def test_selftest_rejects_bad_limits(lib):
    assert lib.pa_selftest_wait_timeout(0, None) == 1
    assert lib.pa_selftest_wait_timeout(6_000_000_000, None) == 1


def test_workspace_size_explicit_partition(lib):
    s = shape(batch=4, max_blocks_per_seq=8192)
    # 131072 tokens in partitions of 512: 256 partitions; acc then (m, l) rows
    n = lib.pa_workspace_size(ctypes.byref(s), 131072, 512)
    rows = 4 * 32 * 256
    acc = rows * 128 * 4
    assert n == (acc + 255) // 256 * 256 + rows * 2 * 4
    assert lib.pa_workspace_size(ctypes.byref(s), 131072, 131072) == 0      # one partition
    assert lib.pa_workspace_size(ctypes.byref(s), 131072, 100) == 0        # not a multiple of 16
    assert lib.pa_workspace_size(ctypes.byref(s), 0, 512) == 0
    # tokens past the table row are not planned for: 16 pages in partitions of 1
    s2 = shape(batch=1, max_blocks_per_seq=16)
    assert lib.pa_workspace_size(ctypes.byref(s2), 10_000, 16) == \
        (1 * 32 * 16 * 128 * 4 + 255) // 256 * 256 + 1 * 32 * 16 * 2 * 4
    # up to 8 partitions reduce inside a thread-block cluster: no workspace
    s3 = shape(batch=1, max_blocks_per_seq=4)
    assert lib.pa_workspace_size(ctypes.byref(s3), 10_000, 16) == 0
    assert lib.pa_workspace_size(ctypes.byref(s), 8 * 512, 512) == 0
    assert lib.pa_workspace_size(ctypes.byref(s), 9 * 512, 512) > 0


@pytest.mark.parametrize("B,T,Hkv", [(1, 512, 8), (16, 256, 8), (4, 2048, 8), (64, 4096, 8),
                                     (1, 131072, 8), (4, 131072, 8), (32, 16384, 1), (2, 60, 8)])
def test_partition_choice_properties(lib, B, T, Hkv):
    H = 32 if Hkv == 8 else 16
    D, bs = (128, 16) if Hkv == 8 else (256, 32)
    s = shape(batch=B, num_heads=H, num_kv_heads=Hkv, head_dim=D, block_size=bs,
              max_blocks_per_seq=(T + bs - 1) // bs)
    for sms in (1, 8, 148, 152):
        pt = lib.pa_choose_partition_tokens(ctypes.byref(s), T, sms)
        assert pt == pa.PARTITION_BALANCED or (pt > 0 and pt % bs == 0)
        assert pt <= ((T + bs - 1) // bs) * bs
    # a grid that already fills the GPU is only cut into partitions of ~64 pages
    pages = (T + bs - 1) // bs
    pt1 = lib.pa_choose_partition_tokens(ctypes.byref(s), T, 1)
    assert pt1 // bs == -(-pages // -(-pages // 64))
    assert lib.pa_choose_partition_tokens(ctypes.byref(s), T, 0) == 0     # invalid SM count


def test_single_sequence_long_context_is_split(lib):
    s = shape(batch=1, max_blocks_per_seq=8192, kv_dtype=pa.BF16)
    pt = lib.pa_choose_partition_tokens(ctypes.byref(s), 131072, 152)
    parts = -(-131072 // pt)
    assert parts * 8 >= 100           # most SMs busy
    assert parts * 8 <= 152           # in a single wave


def test_small_grids_reduce_in_a_cluster(lib):
    # batch 1 x 8 kv heads x 512 tokens: too few pages to balance; 8 partitions in a cluster
    s = shape(batch=1, max_blocks_per_seq=32)
    pt = lib.pa_choose_partition_tokens(ctypes.byref(s), 512, 152)
    assert -(-512 // pt) == 8
    assert lib.pa_workspace_size(ctypes.byref(s), 512, pt) == 0


def test_binding_refuses_cpu_tensors():
    x = torch.zeros(2, 32, 128, dtype=torch.float16)
    with pytest.raises(ValueError):
        pa.decode(torch.zeros(2, 32, 128), x, torch.zeros(8, 16, 8, 128, dtype=torch.float16),
                  torch.zeros(8, 16, 8, 128, dtype=torch.float16),
                  torch.zeros(2, 4, dtype=torch.int32), torch.zeros(2, dtype=torch.int32), 0.1)


def test_plan_info_explicit_partitions(lib):
    """pa_plan_info describes explicit splits without a device."""
    d = pa._PlanDesc()
    s = shape(batch=4, max_blocks_per_seq=8192)
    assert lib.pa_plan_info(ctypes.byref(s), 1, 131072, 512, ctypes.byref(d)) == 0
    assert (d.kernel, d.partitions, d.partition_tokens, d.reduce) == (0, 256, 512, 2)
    assert d.ctas == 4 * 8 * 256
    assert lib.pa_plan_info(ctypes.byref(s), 1, 4096, 512, ctypes.byref(d)) == 0
    assert (d.partitions, d.reduce) == (8, 1)                 # <= 8 partitions: a cluster
    assert lib.pa_plan_info(ctypes.byref(s), 1, 4096, 4096, ctypes.byref(d)) == 0
    assert (d.partitions, d.reduce) == (1, 0)                 # one pass
    # 6 query tokens x group 4 = 24 rows per kv head: the tcgen05 tile kernel
    assert lib.pa_plan_info(ctypes.byref(s), 6, 4096, 1024, ctypes.byref(d)) == 0
    assert (d.kernel, d.partitions, d.threads) == (1, 4, 384)
    assert d.ctas == 4 * 8 * 1 * 4
    # up to 16 rows on the warp-level kernel: query chunks of 16 / group tokens
    assert lib.pa_plan_info(ctypes.byref(s), 4, 4096, 4096, ctypes.byref(d)) == 0
    assert (d.kernel, d.ctas) == (0, 4 * 8)
    assert lib.pa_plan_info(ctypes.byref(s), 0, 4096, 512, ctypes.byref(d)) == 1
    assert lib.pa_plan_info(ctypes.byref(s), 1, 4096, 100, ctypes.byref(d)) == 1
    assert lib.pa_plan_info(ctypes.byref(s), 1, 4096, 512, None) == 1


def test_workspace_size_saturates_instead_of_wrapping(lib):
    """A shape whose partials would need more than a size_t holds reports
    SIZE_MAX (no buffer satisfies it, so the call is refused), never a wrapped
    small size."""
    s = shape(batch=65535, num_heads=65535 * 16, num_kv_heads=65535, head_dim=256,
              max_blocks_per_seq=1 << 26, num_blocks=1000)
    max_ctx = (1 << 30) - 16
    assert lib.pa_workspace_size_multi(ctypes.byref(s), 2000, max_ctx, 16) == 2**64 - 1
    assert lib.pa_workspace_size_multi(ctypes.byref(s), 1, max_ctx, 16) == 2**64 - 1


def test_explicit_plans_and_workspace_sizes_agree(lib):
    """Seeded random shapes and explicit partition sizes, without a device: the
    plan has the requested split, its reduction is a workspace one exactly when
    pa_workspace_size asks for memory, and that size is the layout's
    [B][Hkv][P][Q*G] rows of (D + 2) fp32 (the (m, l) block 256-byte aligned)."""
    rng = np.random.default_rng(7)
    for _ in range(300):
        D = int(rng.choice([64, 128, 256]))
        bs = int(rng.choice([16, 32]))
        G = int(rng.choice([1, 2, 4, 8, 16]))
        Hkv = int(rng.choice([1, 2, 4, 8]))
        B = int(rng.integers(1, 65))
        q_len = int(rng.choice([1, 1, 2, 4, 9, 33]))
        mb = int(rng.integers(1, 2049))
        s = shape(batch=B, num_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                  max_blocks_per_seq=mb, num_blocks=10_000)
        max_ctx = int(rng.integers(0, mb * bs + 1))
        pages = min(-(-max_ctx // bs), mb)
        pp = int(rng.integers(1, 65))
        d = pa._PlanDesc()
        assert lib.pa_plan_info(ctypes.byref(s), q_len, max_ctx, pp * bs, ctypes.byref(d)) == 0
        parts = max(1, -(-pages // pp))
        assert d.partitions == parts
        if parts > 1:
            assert d.partition_tokens == pp * bs
        ws = lib.pa_workspace_size_multi(ctypes.byref(s), q_len, max_ctx, pp * bs)
        assert (ws > 0) == (d.reduce == 2), (d.reduce, ws)
        assert d.reduce in ((0,) if parts == 1 else (1, 2))
        if ws:
            rows = B * G * Hkv * q_len * parts
            assert ws == (rows * D * 4 + 255) // 256 * 256 + rows * 2 * 4


def _binding_args(**over):
    """A consistent set of (CPU) tensors for one decode call, with some replaced."""
    a = dict(out=torch.zeros(2, 32, 128), q=torch.zeros(2, 32, 128, dtype=torch.float16),
             k_cache=torch.zeros(8, 16, 8, 128, dtype=torch.float16),
             v_cache=torch.zeros(8, 16, 8, 128, dtype=torch.float16),
             block_tables=torch.zeros(2, 4, dtype=torch.int32),
             context_lens=torch.zeros(2, dtype=torch.int32))
    a.update(over)
    return a


MISMATCHES = {
    "v_cache_shape": dict(v_cache=torch.zeros(8, 16, 8, 64, dtype=torch.float16)),
    "v_cache_blocks": dict(v_cache=torch.zeros(4, 16, 8, 128, dtype=torch.float16)),
    "v_cache_dtype": dict(v_cache=torch.zeros(8, 16, 8, 128, dtype=torch.bfloat16)),
    "q_dtype": dict(q=torch.zeros(2, 32, 128, dtype=torch.bfloat16)),
    "q_float32": dict(q=torch.zeros(2, 32, 128)),
    "q_head_dim": dict(q=torch.zeros(2, 32, 64, dtype=torch.float16),
                       out=torch.zeros(2, 32, 64)),
    "out_shape": dict(out=torch.zeros(2, 16, 128)),
    "out_dtype": dict(out=torch.zeros(2, 32, 128, dtype=torch.bfloat16)),
    "tables_rows": dict(block_tables=torch.zeros(3, 4, dtype=torch.int32)),
    "lens_rows": dict(context_lens=torch.zeros(3, dtype=torch.int32)),
    "lens_dtype": dict(context_lens=torch.zeros(2, dtype=torch.int64)),
    "tables_dim": dict(block_tables=torch.zeros(8, dtype=torch.int32)),
}


@pytest.mark.parametrize("name", sorted(MISMATCHES))
@pytest.mark.parametrize("entry", ["decode", "decode_splitkv", "decode_splitkv_noalloc"])
def test_binding_refuses_mismatched_tensors(name, entry):
    """Every shape or dtype the library takes on trust is checked by the
    binding before anything reaches the device: the error is the mismatch,
    not the CPU placement of these tensors."""
    a = _binding_args(**MISMATCHES[name])
    fn = getattr(pa, entry)
    extra = () if entry == "decode" else (64,)
    with pytest.raises((ValueError, TypeError)) as e:
        fn(a["out"], a["q"], a["k_cache"], a["v_cache"], a["block_tables"], a["context_lens"],
           0.1, *extra)
    assert "CUDA" not in str(e.value)


def test_binding_refuses_mismatched_multi_token_tensors():
    a = _binding_args(q=torch.zeros(2, 3, 32, 128, dtype=torch.float16), out=torch.zeros(2, 3, 32, 128))
    for over in (dict(out=torch.zeros(2, 2, 32, 128)),
                 dict(v_cache=torch.zeros(8, 16, 8, 128, dtype=torch.bfloat16)),
                 dict(q=torch.zeros(2, 32, 128, dtype=torch.float16))):
        b = dict(a, **over)
        with pytest.raises((ValueError, TypeError)) as e:
            pa.decode_multi(b["out"], b["q"], b["k_cache"], b["v_cache"], b["block_tables"],
                            b["context_lens"], 0.1, 64)
        assert "CUDA" not in str(e.value)


def test_binding_refuses_mismatched_append_and_resolve():
    kc = torch.zeros(8, 16, 8, 128, dtype=torch.float16)
    new = torch.zeros(2, 8, 128, dtype=torch.float16)
    bt = torch.zeros(2, 4, dtype=torch.int32)
    pos = torch.zeros(2, dtype=torch.int32)
    for args in ((kc, torch.zeros(8, 16, 8, 64, dtype=torch.float16), new, new, bt, pos),
                 (kc, kc.clone(), new, new.to(torch.bfloat16), bt, pos),
                 (kc, kc.clone(), new, new, bt, torch.zeros(3, dtype=torch.int32)),
                 (kc, kc.clone(), new[:, :4], new, bt, pos)):
        with pytest.raises((ValueError, TypeError)) as e:
            pa.append_kv(*args)
        assert "CUDA" not in str(e.value)
    with pytest.raises(ValueError) as e:
        pa.resolve_blocks(torch.zeros(2, 4, dtype=torch.int32), bt,
                          torch.zeros(3, dtype=torch.int32), 16, 8)
    assert "CUDA" not in str(e.value)


def test_consistent_cpu_tensors_reach_the_device_check():
    """The validator accepts a consistent set: what stops these CPU tensors is
    the placement check."""
    a = _binding_args()
    with pytest.raises(ValueError, match="CUDA"):
        pa.decode(a["out"], a["q"], a["k_cache"], a["v_cache"], a["block_tables"],
                  a["context_lens"], 0.1)


def test_switches_set_and_restore(lib):
    """The test switches are set through the library (no environment read per
    call); unknown switches and values are refused."""
    k0 = pa.get_switch(pa.SWITCH_MULTI_KERNEL)
    c0 = pa.get_switch(pa.SWITCH_TILE_COMPACT_Q)
    try:
        pa.set_switch(pa.SWITCH_MULTI_KERNEL, pa.KERNEL_TILE)
        assert pa.get_switch(pa.SWITCH_MULTI_KERNEL) == pa.KERNEL_TILE
        pa.set_switch(pa.SWITCH_TILE_COMPACT_Q, 0)
        assert pa.get_switch(pa.SWITCH_TILE_COMPACT_Q) == 0
        with pytest.raises(pa.PaError):
            pa.set_switch(pa.SWITCH_MULTI_KERNEL, 7)
        with pytest.raises(pa.PaError):
            pa.set_switch(pa.SWITCH_TILE_COMPACT_Q, 2)
        with pytest.raises(pa.PaError):
            pa.set_switch(9, 0)
        assert lib.pa_get_switch(9) == -1
        # the kernel switch reaches the plan: 4 rows per kv head on the tile kernel
        s = shape(batch=4, max_blocks_per_seq=256)
        d = pa._PlanDesc()
        assert lib.pa_plan_info(ctypes.byref(s), 1, 4096, 512, ctypes.byref(d)) == 0
        assert d.kernel == 1
        pa.set_switch(pa.SWITCH_MULTI_KERNEL, pa.KERNEL_AUTO)
        assert lib.pa_plan_info(ctypes.byref(s), 1, 4096, 512, ctypes.byref(d)) == 0
        assert d.kernel == 0
    finally:
        pa.set_switch(pa.SWITCH_MULTI_KERNEL, k0)
        pa.set_switch(pa.SWITCH_TILE_COMPACT_Q, c0)


def test_library_reads_no_environment_per_call():
    """The library's source reads the environment only in its load-time
    initialisers."""
    src = open(os.path.join(ROOT, "paged_kv_attention_08_gb300", "csrc", "pa_api.cu")).read()
    assert src.count("getenv") == 1          # inside env_value, used by namespace-scope initialisers
    for f in glob.glob(os.path.join(ROOT, "paged_kv_attention_08_gb300", "csrc", "*")):
        if not f.endswith("pa_api.cu"):
            assert "getenv" not in open(f).read(), f
