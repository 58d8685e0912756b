"""The allocation-free split-KV entry point (pa_decode_splitkv_noalloc).

Some callers cannot allocate device memory -- a host application may hand a
plug-in only fixed input/output buffers, or a latency-critical loop may not
afford cudaMalloc's synchronisation -- so this entry point keeps its partials
in a fixed scratch array inside the library.  These tests call it through the
C ABI twice in a row, on different inputs, and compare each result with the
fp64 CPU oracle and with the workspace entry point (pa_decode_splitkv), both
within the parity tolerance, and check that a call needing more scratch than
the array holds is refused.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_08_gb300 as pa
from paged_kv_attention_08_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = 2e-3
DEV = "cuda:0"


def _out(x):
    return torch.full(x.q.shape, float("nan"), dtype=torch.float32, device=DEV)


def test_noalloc_matches_workspace_entry_point_twice():
    cases = [(workloads.make("sweep_b4_t2048", seed=7, device=DEV), 0),
             (workloads.make("long_b1_t32768", seed=7, device=DEV), 512)]
    refs = [pa.decode_splitkv(_out(x), x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens,
                              x.scale, x.max_context_len, pt) for x, pt in cases]
    # two calls in a row on the same stream, the second on other inputs
    gots = [pa.decode_splitkv_noalloc(_out(x), x.q, x.k_cache, x.v_cache, x.block_tables,
                                      x.context_lens, x.scale, x.max_context_len, pt)
            for x, pt in cases]
    torch.cuda.synchronize()
    for (x, _), ref, got in zip(cases, refs, gots):
        assert torch.isfinite(got).all()
        assert (got - ref).abs().max().item() <= TOL, x.spec.name
        h = x.to("cpu")
        want = oracle.decode_mt(h.q, h.k_cache, h.v_cache, h.block_tables, h.context_lens,
                                h.scale)[0]
        err = np.abs(got.double().cpu().numpy() - want).max()
        assert err <= TOL, f"{x.spec.name}: max abs err {err:.3e} against the oracle"
    assert pa.device_error() == 0


def test_noalloc_refuses_partials_beyond_its_scratch():
    x = workloads.make("long_b1_t32768", seed=8, device=DEV)
    # 2048 partitions of one page: 32 heads x 2048 x 130 floats = 34 MB > 16 MiB
    with pytest.raises(pa.PaError) as ei:
        pa.decode_splitkv_noalloc(_out(x), x.q, x.k_cache, x.v_cache, x.block_tables,
                                  x.context_lens, x.scale, x.max_context_len, 16)
    assert ei.value.code == 3
