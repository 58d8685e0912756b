"""Concurrent calls from several host threads (the C ABI releases the Python
interpreter lock during a call), each on its own stream with its own output
and workspace: every result is bit-identical to the same call made alone.
Covers the library's shared state -- the per-device SM count and error-word
caches, the cluster-occupancy caches, the tensor-map encoder -- under
concurrent first use as far as the process allows, and launches of both
kernels interleaving on the device.
"""
import threading

import pytest
import torch

import paged_kv_attention_08_gb300 as pa
from paged_kv_attention_08_gb300 import workloads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
CALLS = [("sweep_b1_t512", 0), ("sweep_b16_t256", 0), ("sweep_b4_t2048", 0),
         ("sweep_b4_t2048", 256), ("tiny_q8", 0), ("spec_b16_t2048_q4", 0),
         ("chunk_b2_t4096_q64", 0), ("tiny", 32)]


def call(x, pt, stream):
    multi = x.q.dim() == 4
    size = pa.workspace_size_multi if multi else pa.workspace_size
    need = size(x.q, x.k_cache, x.block_tables, torch.float32, x.max_context_len, pt)
    with torch.cuda.stream(stream):
        ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=DEV)
        out = torch.full(x.q.shape, float("nan"), dtype=torch.float32, device=DEV)
    fn = pa.decode_multi if multi else pa.decode_splitkv
    fn(out, x.q, x.k_cache, x.v_cache, x.block_tables, x.context_lens, x.scale,
       x.max_context_len, pt, workspace=ws, stream=stream)
    return out, ws


def test_concurrent_host_threads_bit_identical():
    inputs = [(workloads.make(name, seed=4, device=DEV), pt) for name, pt in CALLS]
    torch.cuda.synchronize()
    n_threads, rounds = 4, 3
    results = [[None] * (len(inputs) * rounds) for _ in range(n_threads)]
    errors = []
    start = threading.Barrier(n_threads)

    def worker(t):
        try:
            stream = torch.cuda.Stream(device=DEV)
            start.wait()
            keep = []
            for r in range(rounds):
                for i in range(len(inputs)):
                    k = (i + t + r) % len(inputs)   # threads interleave different calls
                    x, pt = inputs[k]
                    out, ws = call(x, pt, stream)
                    keep.append(ws)
                    results[t][r * len(inputs) + i] = (k, out)
            stream.synchronize()
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(n_threads)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
    assert not any(th.is_alive() for th in threads), "a worker did not finish"
    assert not errors, errors
    torch.cuda.synchronize()
    alone = []
    for x, pt in inputs:
        out, _ = call(x, pt, torch.cuda.current_stream())
        torch.cuda.synchronize()
        alone.append(out)
    for t in range(n_threads):
        for k, out in results[t]:
            assert torch.equal(out, alone[k]), f"thread {t}, call {CALLS[k]}"
    assert pa.device_error() == 0
