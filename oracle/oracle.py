"""Python front end of the C oracle (``oracle.c``) for the verify step.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` are the only callers. The CUDA path
and its binding never import this module.

Everything here is argument marshalling (numpy arrays to pointers) plus a
thread pool over disjoint sequence ranges; all of the verify arithmetic lives
in ``oracle.c`` and follows the pages cited there. The LM-head logits use a
float64 matrix product (a library primitive) over exactly widened bf16 values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, BF16, F64 = 0, 1, 2
GREEDY, SAMPLE = 0, 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain gcc, IEEE arithmetic)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"],
                       check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str):
    """Load a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    lib.oracle_verify.restype = ctypes.c_int
    lib.oracle_verify.argtypes = [
        P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_double, P, ctypes.c_uint64, P, P, ctypes.c_int, ctypes.c_int,
        P, P, P, P, P, P, P, P, P, P]
    lib.oracle_verify_tree.restype = ctypes.c_int
    lib.oracle_verify_tree.argtypes = [P, ctypes.c_int, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, P, P, P]
    lib.oracle_prompt_lookup.restype = None
    lib.oracle_prompt_lookup.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, P, P]
    lib.oracle_philox4x32_10.restype = None
    lib.oracle_philox4x32_10.argtypes = [P, P, P]
    lib.oracle_philox_uniforms.restype = None
    lib.oracle_philox_uniforms.argtypes = [ctypes.c_uint64, P, ctypes.c_int, ctypes.c_int,
                                           P, P]
    lib.oracle_lmhead_logits.restype = None
    lib.oracle_lmhead_logits.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, P]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:  # raw bf16 bits
        return BF16
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"logits must be float32, float64 or uint16 (bf16 bits), got {a.dtype}")


def philox4x32_10(counter, key) -> np.ndarray:
    lib = _load()
    c = np.ascontiguousarray(counter, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib.oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def philox_uniforms(seed: int, seq_ids, n_pos: int):
    """(u, u2) arrays [len(seq_ids), n_pos] of the draws used by the verify step."""
    lib = _load()
    ids = np.ascontiguousarray(seq_ids, dtype=np.uint64)
    u = np.zeros((ids.size, n_pos))
    u2 = np.zeros((ids.size, n_pos))
    lib.oracle_philox_uniforms(ctypes.c_uint64(seed), _ptr(ids), ids.size, n_pos, _ptr(u), _ptr(u2))
    return u, u2


def verify(target, draft, draft_tokens, temperature=1.0, modes=SAMPLE, seed=0, seq_ids=None,
           uniforms=None, threads=1, seq_range=None, draft_lens=None):
    """Run the oracle verify step.

    target [B, K+1, V] and draft [B, K, V]: float32, float64 or uint16 (bf16
    bits); draft may be None when every sequence is greedy. draft_tokens
    [B, K] int. modes: 0/1 or an array [B]. uniforms: optional (u, u2), each
    [B, K+1], replacing the Philox draws. seq_range=(b0, b1) restricts the
    work to those sequences (the other outputs stay at their fill values).
    draft_lens: optional [B] ints, sequence b verifying only its first
    draft_lens[b] drafts (0..K; other values make it invalid).
    Returns a dict of numpy arrays.
    """
    lib = _load()
    target = np.ascontiguousarray(target)
    B, K1, V = target.shape
    K = K1 - 1
    tokens = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, K)
    modes_arr = np.ascontiguousarray(np.broadcast_to(np.asarray(modes, dtype=np.int32), (B,)))
    if draft is not None:
        draft = np.ascontiguousarray(draft)
        assert draft.shape == (B, K, V)
        dtype_d = _dtype_code(draft)
    else:
        assert not modes_arr.any(), "sample mode needs draft logits"
        dtype_d = F32
    ids = None if seq_ids is None else np.ascontiguousarray(seq_ids, dtype=np.uint64)
    lens = None if draft_lens is None else np.ascontiguousarray(draft_lens, dtype=np.int32).reshape(B)
    uni = None
    if uniforms is not None:
        uni = np.ascontiguousarray(np.stack([np.asarray(uniforms[0], dtype=np.float64).reshape(B, K1),
                                             np.asarray(uniforms[1], dtype=np.float64).reshape(B, K1)]))
    out = {
        "tokens": np.full((B, K1), -1, dtype=np.int32),
        "n_accepted": np.full(B, -2, dtype=np.int32),
        "p_target": np.full((B, K), np.nan),
        "p_draft": np.full((B, K), np.nan),
        "residual_mass": np.full(B, np.nan),
        "accept_margin": np.full(B, np.inf),
        "draw_margin": np.full(B, np.inf),
        "draw_edges": np.full((B, 2), np.nan),
        "fallback": np.zeros(B, dtype=np.int32),
    }
    b0, b1 = (0, B) if seq_range is None else seq_range

    def run(lo, hi):
        rc = lib.oracle_verify(
            _ptr(target), _ptr(draft), _ptr(tokens), B, K, V, _dtype_code(target), dtype_d,
            float(temperature), _ptr(modes_arr), ctypes.c_uint64(seed), _ptr(ids), _ptr(uni),
            lo, hi, _ptr(out["tokens"]), _ptr(out["n_accepted"]), _ptr(out["p_target"]),
            _ptr(out["p_draft"]), _ptr(out["residual_mass"]), _ptr(out["accept_margin"]),
            _ptr(out["draw_margin"]), _ptr(out["fallback"]), _ptr(lens), _ptr(out["draw_edges"]))
        if rc != 0:
            raise MemoryError("oracle_verify could not allocate its work buffers")

    threads = max(1, min(int(threads), b1 - b0))
    if threads == 1:
        run(b0, b1)
    else:
        bounds = np.linspace(b0, b1, threads + 1).astype(int)
        with ThreadPoolExecutor(threads) as pool:
            list(pool.map(lambda i: run(bounds[i], bounds[i + 1]), range(threads)))
    return out


def verify_tree(target, tokens, parents):
    """Greedy tree verification. target [B, N, V] (float32, float64 or bf16
    bits), tokens and parents [B, N] (parents[b, 0] is ignored: node 0 is the
    root). Returns dict(tokens [B, N], n_accepted [B], last_node [B])."""
    lib = _load()
    target = np.ascontiguousarray(target)
    B, N, V = target.shape
    tok = np.ascontiguousarray(np.broadcast_to(np.asarray(tokens, dtype=np.int32), (B, N)))
    par = np.ascontiguousarray(np.broadcast_to(np.asarray(parents, dtype=np.int32), (B, N)))
    out = {"tokens": np.full((B, N), -1, dtype=np.int32), "n_accepted": np.full(B, -2, dtype=np.int32),
           "last_node": np.full(B, -2, dtype=np.int32)}
    rc = lib.oracle_verify_tree(_ptr(target), _dtype_code(target), _ptr(tok), _ptr(par), B, N, V, 0, B,
                                _ptr(out["tokens"]), _ptr(out["n_accepted"]), _ptr(out["last_node"]))
    if rc != 0:
        raise MemoryError("oracle_verify_tree could not allocate its work buffers")
    return out


def prompt_lookup(tokens, lengths, max_ngram=3, n_drafts=5):
    """Prompt lookup drafting. tokens [B, L_max] int, lengths [B] int.
    Returns dict(drafts [B, n_drafts] (-1 padded), n_drafts [B])."""
    lib = _load()
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    B, L_max = tok.shape
    lens = np.ascontiguousarray(np.broadcast_to(np.asarray(lengths, dtype=np.int32), (B,)))
    out = {"drafts": np.full((B, n_drafts), -1, dtype=np.int32), "n_drafts": np.full(B, -2, dtype=np.int32)}
    lib.oracle_prompt_lookup(_ptr(tok), _ptr(lens), B, L_max, int(max_ngram), int(n_drafts), 0, B,
                             _ptr(out["drafts"]), _ptr(out["n_drafts"]))
    return out


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of raw bf16 bits (uint16) to float64."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def lmhead_logits(hidden_bits: np.ndarray, w_bits: np.ndarray, rows=None, v_chunk: int = 8192,
                  use_c: bool = False) -> np.ndarray:
    """float64 logits[rows, V] = hidden[rows] @ W over exactly widened bf16.

    hidden_bits [M, d] and w_bits [d, V] are raw bf16 bits (uint16). The
    default uses a float64 matrix product over V chunks; use_c=True runs the
    plain C triple loop instead (slow; for small shapes and for checking the
    two against each other)."""
    hidden_bits = np.ascontiguousarray(hidden_bits, dtype=np.uint16)
    w_bits = np.ascontiguousarray(w_bits, dtype=np.uint16)
    M, d = hidden_bits.shape
    d2, V = w_bits.shape
    assert d == d2
    rows = np.arange(M) if rows is None else np.asarray(rows)
    if use_c:
        lib = _load()
        out = np.zeros((len(rows), V))
        for i, m in enumerate(rows):
            lib.oracle_lmhead_logits(_ptr(hidden_bits), _ptr(w_bits), M, d, V, int(m), int(m) + 1,
                                     out[i:].ctypes.data)
        return out
    h = bf16_to_f64(hidden_bits[rows])
    out = np.empty((len(rows), V))
    for v0 in range(0, V, v_chunk):
        out[:, v0:v0 + v_chunk] = h @ bf16_to_f64(w_bits[:, v0:v0 + v_chunk])
    return out
