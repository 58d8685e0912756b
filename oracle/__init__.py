"""fp64 CPU oracle for paged-attention decode.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (``paged_kv_attention_08_gb300``) never imports it and shares no
code with it; the two meet only in the seeded input generator, which holds none
of the method's arithmetic.

The arithmetic lives in ``pa_oracle.c`` (plain C, fp64, one block-table lookup
per token; see that file's header for the passages it follows and the readings
it takes).  This module compiles it with gcc on first use and marshals torch /
numpy arrays into it.

Parity status of each function (pins live in ``tests/test_oracle_pins.py``):
  decode, decode_rows  -- pinned: closed forms (single token, equal keys, one
                          dominant score, a hand-worked two-token case), dense
                          brute force, torch SDPA special case, pool-permutation
                          invariance, masking semantics.
  resolve_blocks       -- pinned: brute force over an independent per-page rule
                          and hand-written cases.
  decode_multi         -- pinned: each query row equals the one-token decode of
                          its causal prefix (bit-exact), q_len = 1 equals
                          decode, dense brute force with an explicit causal mask.
  append_kv            -- pinned: exactly the addressed slots change (element
                          by element over the whole pool), invalid positions and
                          entries write nothing, append-then-decode equals the
                          decode of a cache built with the token in place.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpa_oracle.so")

_lock = threading.Lock()
_lib = None

F16, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile ``pa_oracle.c`` into ``oracle/_build/libpa_oracle.so`` with gcc."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.run(
            ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # PA_ORACLE_LIB lets the mutation test load a deliberately broken
            # copy of the oracle to prove that the pins catch it.
            lib = ctypes.CDLL(os.environ.get("PA_ORACLE_LIB") or build())
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.pao_decode.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, i32, f64]
            lib.pao_decode.restype = ctypes.c_int
            lib.pao_decode_rows.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64,
                                            i32, f64, P, i32]
            lib.pao_decode_rows.restype = ctypes.c_int
            lib.pao_resolve_blocks.argtypes = [P, P, P, i32, i32, i32, i64]
            lib.pao_resolve_blocks.restype = ctypes.c_int
            lib.pao_decode_multi.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                             i64, i32, f64]
            lib.pao_decode_multi.restype = ctypes.c_int
            lib.pao_append_kv.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i64]
            lib.pao_append_kv.restype = ctypes.c_int
            _lib = lib
    return _lib


def _u16(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit patterns of an fp16/bf16 tensor, on the host, contiguous."""
    if t.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError(f"oracle takes fp16/bf16 inputs, got {t.dtype}")
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _i32(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(t, dtype=np.int32))


def _dtype_code(t: torch.Tensor) -> int:
    return BF16 if t.dtype == torch.bfloat16 else F16


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _common(q, k_cache, v_cache, block_tables, context_lens):
    if q.dtype != k_cache.dtype or k_cache.dtype != v_cache.dtype:
        raise TypeError("q, k_cache and v_cache must share one dtype")
    B, H, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    if D2 != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("cache shape does not match q")
    bt = _i32(block_tables)
    if bt.ndim != 2 or bt.shape[0] != B:
        raise ValueError("block_tables must be [batch, max_blocks]")
    lens = _i32(context_lens)
    if lens.shape != (B,):
        raise ValueError("context_lens must be [batch]")
    return (B, H, Hkv, D, bs, bt.shape[1], NB), bt, lens


def decode(q, k_cache, v_cache, block_tables, context_lens, scale: float) -> np.ndarray:
    """out[b, h, :] in float64 for every sequence and query head.

    ``scale`` is rounded to fp32 first: the decode library takes it as a C
    float, so that fp32 value is the input both sides compute with.
    """
    (B, H, Hkv, D, bs, mb, NB), bt, lens = _common(q, k_cache, v_cache, block_tables, context_lens)
    qa, ka, va = _u16(q), _u16(k_cache), _u16(v_cache)
    out = np.zeros((B, H, D), dtype=np.float64)
    rc = _load().pao_decode(_ptr(out), _ptr(qa), _ptr(ka), _ptr(va), _ptr(bt), _ptr(lens),
                            B, H, Hkv, D, bs, mb, NB, _dtype_code(q), float(np.float32(scale)))
    if rc != 0:
        raise RuntimeError("oracle decode rejected its arguments")
    return out


def decode_rows(q, k_cache, v_cache, block_tables, context_lens, scale: float, rows) -> np.ndarray:
    """out for selected (b, h) pairs only: ``rows`` is an [n, 2] int array."""
    (B, H, Hkv, D, bs, mb, NB), bt, lens = _common(q, k_cache, v_cache, block_tables, context_lens)
    rows = _i32(rows).reshape(-1, 2)
    qa, ka, va = _u16(q), _u16(k_cache), _u16(v_cache)
    out = np.zeros((rows.shape[0], D), dtype=np.float64)
    rc = _load().pao_decode_rows(_ptr(out), _ptr(qa), _ptr(ka), _ptr(va), _ptr(bt), _ptr(lens),
                                 B, H, Hkv, D, bs, mb, NB, _dtype_code(q),
                                 float(np.float32(scale)), _ptr(rows), rows.shape[0])
    if rc != 0:
        raise RuntimeError("oracle decode_rows rejected its arguments")
    return out


def host_threads() -> int:
    """Host cores this process may run on (its CPU affinity)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return max(1, os.cpu_count() or 1)


def decode_mt(q, k_cache, v_cache, block_tables, context_lens, scale: float,
              threads: int | None = None) -> tuple[np.ndarray, int]:
    """``decode``'s result computed on several host threads: the (sequence,
    head) rows are cut into one contiguous chunk per thread and each chunk goes
    through ``pao_decode_rows`` -- the same per-row arithmetic as ``decode``,
    run side by side (the foreign calls release the interpreter lock).  For
    timing the oracle on all the host's cores.  Returns (out, threads used)."""
    (B, H, Hkv, D, bs, mb, NB), bt, lens = _common(q, k_cache, v_cache, block_tables, context_lens)
    qa, ka, va = _u16(q), _u16(k_cache), _u16(v_cache)
    n = B * H
    threads = max(1, min(threads or host_threads(), n)) if n else 1
    rows = np.stack(np.meshgrid(np.arange(B, dtype=np.int32), np.arange(H, dtype=np.int32),
                                indexing="ij"), axis=-1).reshape(-1, 2).copy()
    out = np.zeros((n, D), dtype=np.float64)
    bounds = [n * i // threads for i in range(threads + 1)]
    lib = _load()
    dt, sc = _dtype_code(q), float(np.float32(scale))
    rcs = [0] * threads

    def run(i):
        lo, hi = bounds[i], bounds[i + 1]
        if hi > lo:
            r = np.ascontiguousarray(rows[lo:hi])
            o = np.zeros((hi - lo, D), dtype=np.float64)
            rcs[i] = lib.pao_decode_rows(_ptr(o), _ptr(qa), _ptr(ka), _ptr(va), _ptr(bt),
                                         _ptr(lens), B, H, Hkv, D, bs, mb, NB, dt, sc, _ptr(r),
                                         hi - lo)
            out[lo:hi] = o

    workers = [threading.Thread(target=run, args=(i,)) for i in range(threads)]
    for w in workers:
        w.start()
    for w in workers:
        w.join()
    if any(rcs):
        raise RuntimeError("oracle decode_rows rejected its arguments")
    return out.reshape(B, H, D), threads


def resolve_blocks(block_tables, context_lens, block_size: int, num_blocks: int) -> np.ndarray:
    """[batch, max_blocks] int32: the physical block read for each logical page,
    -1 where the page holds no attended token."""
    bt = _i32(block_tables)
    lens = _i32(context_lens)
    B, mb = bt.shape
    out = np.full((B, mb), -1, dtype=np.int32)
    rc = _load().pao_resolve_blocks(_ptr(out), _ptr(bt), _ptr(lens), B, block_size, mb, num_blocks)
    if rc != 0:
        raise RuntimeError("oracle resolve_blocks rejected its arguments")
    return out


def append_kv(k_cache, v_cache, k_new, v_new, block_tables, positions):
    """New k_cache, v_cache (copies) with each sequence's token written at its
    position's slot; k_new, v_new are [batch, num_kv_heads, head_dim]."""
    if k_new.dtype != k_cache.dtype or v_new.dtype != v_cache.dtype:
        raise TypeError("new keys/values must have the cache's dtype")
    NB, bs, Hkv, D = k_cache.shape
    bt = _i32(block_tables)
    pos = _i32(positions)
    B, mb = bt.shape
    if tuple(k_new.shape) != (B, Hkv, D) or tuple(v_new.shape) != (B, Hkv, D) or pos.shape != (B,):
        raise ValueError("k_new/v_new must be [batch, num_kv_heads, head_dim], positions [batch]")
    ka, va = _u16(k_cache).copy(), _u16(v_cache).copy()
    kn, vn = _u16(k_new), _u16(v_new)
    rc = _load().pao_append_kv(_ptr(ka), _ptr(va), _ptr(kn), _ptr(vn), _ptr(bt), _ptr(pos),
                               B, Hkv, D, bs, mb, NB)
    if rc != 0:
        raise RuntimeError("oracle append_kv rejected its arguments")
    to_t = lambda a: torch.from_numpy(a.view(np.int16).reshape(NB, bs, Hkv, D)).view(k_cache.dtype)
    return to_t(ka), to_t(va)


def decode_multi(q, k_cache, v_cache, block_tables, context_lens, scale: float) -> np.ndarray:
    """Several query tokens per sequence: q [B, Q, H, D] -> out [B, Q, H, D]
    float64; query token i attends causally to tokens <= T - Q + i."""
    if q.dim() != 4:
        raise ValueError("q must be [batch, q_len, num_heads, head_dim]")
    B, Q, H, D = q.shape
    (_, _, Hkv, _, bs, mb, NB), bt, lens = _common(q[:, 0], k_cache, v_cache, block_tables,
                                                  context_lens)
    qa, ka, va = _u16(q), _u16(k_cache), _u16(v_cache)
    out = np.zeros((B, Q, H, D), dtype=np.float64)
    rc = _load().pao_decode_multi(_ptr(out), _ptr(qa), _ptr(ka), _ptr(va), _ptr(bt), _ptr(lens),
                                  B, Q, H, Hkv, D, bs, mb, NB, _dtype_code(q),
                                  float(np.float32(scale)))
    if rc != 0:
        raise RuntimeError("oracle decode_multi rejected its arguments")
    return out


def decode_multi_mt(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                    threads: int | None = None) -> tuple[np.ndarray, int]:
    """``decode_multi``'s result computed on several host threads, for timing
    and for checking whole outputs quickly.  The work is cut into pieces of
    (one sequence, a run of its query tokens): the run [i0, i1) of sequence b
    is a multi-token decode of its own -- q_len = i1 - i0 query tokens whose
    last sits at position T - Q + i1 - 1, i.e. a context length of
    T - Q + i1 -- so each piece goes through ``pao_decode_multi`` unchanged
    (same per-row arithmetic, the cache shared and read only).  Returns
    (out, threads used)."""
    if q.dim() != 4:
        raise ValueError("q must be [batch, q_len, num_heads, head_dim]")
    B, Q, H, D = q.shape
    (_, _, Hkv, _, bs, mb, NB), bt, lens = _common(q[:, 0], k_cache, v_cache, block_tables,
                                                  context_lens)
    qa, ka, va = _u16(q), _u16(k_cache), _u16(v_cache)
    out = np.zeros((B, Q, H, D), dtype=np.float64)
    want = max(1, threads or host_threads())
    # enough pieces that every thread gets some: split each sequence's query
    # tokens into ceil(want / B) runs
    runs = max(1, min(Q, -(-want // B))) if B else 1
    pieces = [(b, Q * r // runs, Q * (r + 1) // runs) for b in range(B) for r in range(runs)]
    pieces = [p for p in pieces if p[2] > p[1]]
    threads = max(1, min(want, len(pieces))) if pieces else 1
    lib = _load()
    dt, sc = _dtype_code(q), float(np.float32(scale))
    rcs = [0] * len(pieces)
    nxt = [0]
    lock = threading.Lock()

    def run():
        while True:
            with lock:
                k = nxt[0]
                nxt[0] += 1
            if k >= len(pieces):
                return
            b, i0, i1 = pieces[k]
            qs = np.ascontiguousarray(qa[b:b + 1, i0:i1])
            bts = np.ascontiguousarray(bt[b:b + 1])
            ls = np.array([int(lens[b]) - Q + i1], dtype=np.int32)
            o = np.zeros((1, i1 - i0, H, D), dtype=np.float64)
            rcs[k] = lib.pao_decode_multi(_ptr(o), _ptr(qs), _ptr(ka), _ptr(va), _ptr(bts),
                                          _ptr(ls), 1, i1 - i0, H, Hkv, D, bs, mb, NB, dt, sc)
            out[b, i0:i1] = o[0]

    workers = [threading.Thread(target=run) for _ in range(threads)]
    for w in workers:
        w.start()
    for w in workers:
        w.join()
    if any(rcs):
        raise RuntimeError("oracle decode_multi rejected its arguments")
    return out, threads


def cpu_model() -> str:
    """The host CPU's name as /proc/cpuinfo gives it (model name, or the Arm
    implementer and part numbers), else the machine type."""
    import platform
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        info = []
    for ln in info:
        if ln.lower().startswith("model name"):
            return ln.split(":", 1)[1].strip()
    impl = next((ln.split(":", 1)[1].strip() for ln in info if ln.startswith("CPU implementer")), None)
    part = next((ln.split(":", 1)[1].strip() for ln in info if ln.startswith("CPU part")), None)
    if impl and part:
        return f"{platform.machine()} (CPU implementer {impl}, part {part})"
    return platform.machine() or "unknown"

