"""Seeded synthetic inputs for paged-attention decode.

This module only draws random numbers and lays them out; it holds none of the
decode arithmetic, so both the CUDA path and the CPU oracle may take their
inputs from it.

Shapes and distributions follow the benchmark set-up on the pages:
  - "benchmark_decoding.py", setup_test_data: q ~ N(0,1) of shape
    [batch, num_heads, head_dim]; k_cache / v_cache ~ N(0,1) of shape
    [num_blocks, block_size, num_kv_heads, head_dim]; the block table is a
    seeded random permutation of the pool (not arange, so that a kernel which
    ignores the table cannot pass); scale = 1/sqrt(head_dim).
  - MiniVLLM docs "Decoding Benchmark", table "Benchmark configurations": the
    (batch, seq_len) sweep with 32 query heads, 8 kv heads, head_dim 128 and
    block_size 16.
plus the ragged, long-context and MQA workloads this library is measured on,
and multi-token steps (q_len > 1: speculative verification of drafted
tokens, a short chunk of new tokens) whose query is [batch, q_len,
num_heads, head_dim] and whose context lengths count the new tokens.

Recipe (identical for every workload):
  1. The index structure (context lengths, block tables) is drawn on the CPU
     from ``torch.Generator().manual_seed(seed)``, so it does not depend on the
     device.
  2. Lengths are fixed, or uniform integers in [lo, hi].
  3. The pool holds exactly the needed pages ("exact"), a multiple of them
     rounded up ("factor"), or a fixed count.  A seeded ``randperm`` of the pool
     is dealt out page by page to the sequences in order, so used blocks are
     scattered and any spare ones are interleaved among them; the rest of each
     table row is -1.
  4. Values (q, then K, then V) are drawn as fp32 N(0,1) from a generator on
     the target device seeded with ``seed + 1``, multiplied by the workload's
     standard deviation and rounded to fp16/bf16 (round to nearest even).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Spec:
    name: str
    batch: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: torch.dtype
    lens: str                 # "fixed:T", "list:a,b,...", "uniform:lo:hi"
    pool: str = "exact"       # "exact", "factor:F", "fixed:N"
    max_blocks: int = 0       # 0: the largest number of pages any sequence needs
    q_std: float = 1.0
    kv_std: float = 1.0
    partition_tokens: int = 0  # split-KV partition size this workload runs with (0: automatic)
    q_len: int = 1             # query tokens per sequence (q is [B, H, D] when 1, else [B, Q, H, D])


def _sweep(b, t):
    return Spec(f"sweep_b{b}_t{t}", b, 32, 8, 128, 16, torch.float16, f"fixed:{t}")


def _long(b, t):
    return Spec(f"long_b{b}_t{t}", b, 32, 8, 128, 16, torch.bfloat16, f"fixed:{t}",
                partition_tokens=512)


SPECS = {s.name: s for s in [
    # two sequences of 60 tokens in a pool of 8 blocks, 4 table slots each
    Spec("tiny", 2, 32, 8, 128, 16, torch.float16, "list:60,60", pool="fixed:8", max_blocks=4),
    _sweep(1, 512), _sweep(16, 256), _sweep(4, 2048),
    Spec("ragged_b64", 64, 32, 8, 128, 16, torch.bfloat16, "uniform:1:4096", pool="factor:1.25",
         max_blocks=256),
    _long(1, 8192), _long(1, 32768), _long(1, 131072),
    _long(4, 8192), _long(4, 32768), _long(4, 131072),
    Spec("mqa_b32_t16384", 32, 16, 1, 256, 32, torch.bfloat16, "fixed:16384", pool="factor:1.1",
         q_std=1.0, kv_std=0.5),
    # the MQA shape at smoke-test size: 3 + 5 pages of 32 tokens, one spare block
    Spec("tiny_mqa", 2, 16, 1, 256, 32, torch.bfloat16, "list:70,130", pool="fixed:9",
         max_blocks=5, kv_std=0.5),
    # multi-token steps: a small case with a sequence shorter than q_len, four
    # drafted tokens per sequence (4 tokens x 4 heads fill the 16 MMA rows),
    # eight (two CTAs per kv head), and a 64-token chunk with MQA-like groups
    Spec("tiny_q3", 3, 32, 8, 128, 16, torch.float16, "list:2,37,60", pool="fixed:12",
         max_blocks=4, q_len=3),
    # 8 query tokens x 4 heads = 32 rows per kv head: the tcgen05 tile kernel
    Spec("tiny_q8", 2, 32, 8, 128, 16, torch.bfloat16, "list:40,70", pool="fixed:9",
         max_blocks=5, q_len=8),
    Spec("spec_b16_t2048_q4", 16, 32, 8, 128, 16, torch.float16, "fixed:2048", q_len=4),
    Spec("spec_b4_t8192_q8", 4, 32, 8, 128, 16, torch.bfloat16, "fixed:8192", q_len=8),
    Spec("chunk_b2_t4096_q64", 2, 16, 1, 256, 32, torch.bfloat16, "fixed:4096", pool="factor:1.1",
         kv_std=0.5, q_len=64),
    # a 256-token chunk on the GQA shape: 1024 rows per kv head, eight 128-row tiles
    Spec("prefill_b16_t2048_q256", 16, 32, 8, 128, 16, torch.float16, "fixed:2048", q_len=256),
]}

# Named groups of workloads; a group is run as a sequence of decode calls.
GROUPS = {
    "tiny": ["tiny"],
    "sweep": ["sweep_b1_t512", "sweep_b16_t256", "sweep_b4_t2048"],
    "ragged": ["ragged_b64"],
    "long": ["long_b1_t8192", "long_b1_t32768", "long_b1_t131072",
             "long_b4_t8192", "long_b4_t32768", "long_b4_t131072"],
    "mqa": ["mqa_b32_t16384"],
    "multi": ["spec_b16_t2048_q4", "spec_b4_t8192_q8", "chunk_b2_t4096_q64"],
}
# every single workload is also a group of its own
GROUPS.update({name: [name] for name in SPECS if name not in GROUPS})


@dataclass
class Inputs:
    spec: Spec
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_tables: torch.Tensor   # int32 [batch, max_blocks], -1 padded
    context_lens: torch.Tensor   # int32 [batch]
    scale: float
    max_context_len: int
    lens_host: list = field(default_factory=list)

    @property
    def num_blocks(self) -> int:
        return self.k_cache.shape[0]

    def to(self, device) -> "Inputs":
        return Inputs(self.spec, self.q.to(device), self.k_cache.to(device), self.v_cache.to(device),
                      self.block_tables.to(device), self.context_lens.to(device), self.scale,
                      self.max_context_len, list(self.lens_host))


def _draw_lens(spec: Spec, g: torch.Generator) -> list:
    kind, _, rest = spec.lens.partition(":")
    if kind == "fixed":
        return [int(rest)] * spec.batch
    if kind == "list":
        lens = [int(x) for x in rest.split(",")]
        assert len(lens) == spec.batch
        return lens
    if kind == "uniform":
        lo, hi = (int(x) for x in rest.split(":"))
        return torch.randint(lo, hi + 1, (spec.batch,), generator=g).tolist()
    raise ValueError(spec.lens)


def _pool_size(spec: Spec, needed: int) -> int:
    kind, _, rest = spec.pool.partition(":")
    if kind == "exact":
        return needed
    if kind == "factor":
        return int(math.ceil(float(rest) * needed))
    if kind == "fixed":
        n = int(rest)
        assert n >= needed
        return n
    raise ValueError(spec.pool)


def _randn_into(out: torch.Tensor, std: float, g: torch.Generator, chunk_elems: int = 1 << 26):
    """Fill ``out`` (fp16/bf16) with N(0, std^2) drawn in fp32, chunk by chunk."""
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        x = torch.randn(e - s, generator=g, device=out.device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        flat[s:e].copy_(x)


def make(spec, seed: int = 0, device="cpu") -> Inputs:
    """Build the seeded inputs of one workload (a ``Spec`` or its name)."""
    if isinstance(spec, str):
        spec = SPECS[spec]
    device = torch.device(device)
    gi = torch.Generator().manual_seed(seed)
    lens = _draw_lens(spec, gi)
    bs = spec.block_size
    pages = [(t + bs - 1) // bs for t in lens]
    max_blocks = spec.max_blocks or max(1, max(pages))
    assert max(pages) <= max_blocks, "a sequence needs more pages than its table row holds"
    needed = sum(pages)
    pool = max(1, _pool_size(spec, needed))
    perm = torch.randperm(pool, generator=gi, dtype=torch.int64)
    table = torch.full((spec.batch, max_blocks), -1, dtype=torch.int32)
    cursor = 0
    for b, n in enumerate(pages):
        table[b, :n] = perm[cursor:cursor + n].to(torch.int32)
        cursor += n

    gv = torch.Generator(device=device).manual_seed(seed + 1)
    qshape = (spec.batch, spec.num_heads, spec.head_dim) if spec.q_len == 1 else \
        (spec.batch, spec.q_len, spec.num_heads, spec.head_dim)
    q = torch.empty(qshape, dtype=spec.dtype, device=device)
    k = torch.empty(pool, bs, spec.num_kv_heads, spec.head_dim, dtype=spec.dtype, device=device)
    v = torch.empty_like(k)
    _randn_into(q, spec.q_std, gv)
    _randn_into(k, spec.kv_std, gv)
    _randn_into(v, spec.kv_std, gv)
    return Inputs(spec, q, k, v, table.to(device), torch.tensor(lens, dtype=torch.int32, device=device),
                  1.0 / math.sqrt(spec.head_dim), max(lens) if lens else 0, list(lens))
