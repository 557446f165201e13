"""Thin ctypes binding of libspecverify (argument marshalling only).

Every function takes torch tensors that already live on the current CUDA
device, passes their data pointers and the current torch stream to the C ABI
declared in include/specverify.h, and raises SpecVerifyError on a non-OK
status. All of the verify arithmetic runs in the library's CUDA kernels; this
module computes nothing. Missing outputs are allocated with torch.empty.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspecverify.so")
DEBUG_LIB_PATH = os.path.join(_PKG, "libspecverify_debug.so")

SV_F32, SV_BF16 = 0, 1
SV_GREEDY, SV_SAMPLE = 0, 1

SV_FLAG_BAD_TOKEN = 1
SV_FLAG_BAD_ROW = 2
SV_FLAG_RESIDUAL_FALLBACK = 4
SV_FLAG_DRAW_EDGE = 8
SV_FLAG_BAD_MODE = 16
SV_FLAG_TIMEOUT = 32
SV_FLAG_BAD_LENGTH = 64
SV_FLAG_BAD_TREE = 128
SV_FLAG_DEBUG_BOUNDS = 256
SV_ARG_OVERLAP_PREVIOUS = 1
SV_ARG_TEST_WAIT_TIMEOUT = 0x80000000
SV_ARG_TEST_DEBUG_SHRINK = 0x40000000
SV_ERR_SCRATCH_LIMIT = 12
SV_LMHEAD_SCRATCH_BYTES = 32 << 20  # include/specverify.h

STATUS_NAMES = {
    0: "SV_OK", 1: "SV_ERR_NULL", 2: "SV_ERR_SHAPE", 3: "SV_ERR_DTYPE", 4: "SV_ERR_TEMPERATURE",
    5: "SV_ERR_WORKSPACE", 6: "SV_ERR_ARCH", 7: "SV_ERR_CUDA", 8: "SV_ERR_MODE",
    9: "SV_ERR_ALIGN", 10: "SV_ERR_CONFIG", 11: "SV_ERR_NOT_IMPLEMENTED",
}


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {STATUS_NAMES.get(status, status)} ({sv_status_string(status)})"
        if status == 7:
            msg += f"; cuda error {_load().sv_last_cuda_error()}"
        super().__init__(msg)


class sv_verify_args(ctypes.Structure):
    """Mirror of sv_verify_args in include/specverify.h."""
    _fields_ = [
        ("target_logits", ctypes.c_void_p),
        ("draft_logits", ctypes.c_void_p),
        ("draft_tokens", ctypes.c_void_p),
        ("B", ctypes.c_int),
        ("K", ctypes.c_int),
        ("V", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("temperature", ctypes.c_float),
        ("mode", ctypes.c_int),
        ("modes", ctypes.c_void_p),
        ("seed", ctypes.c_uint64),
        ("seq_ids", ctypes.c_void_p),
        ("out_tokens", ctypes.c_void_p),
        ("out_n_accepted", ctypes.c_void_p),
        ("out_p_target", ctypes.c_void_p),
        ("out_p_draft", ctypes.c_void_p),
        ("out_residual_mass", ctypes.c_void_p),
        ("status_word", ctypes.c_void_p),
        ("cluster_size", ctypes.c_int),
        ("stream", ctypes.c_void_p),
        ("flags", ctypes.c_uint32),
        ("draft_lens", ctypes.c_void_p),
        ("out_draw_edges", ctypes.c_void_p),
        ("seqs_per_cluster", ctypes.c_int),
    ]


class sv_verify_plan(ctypes.Structure):
    """Mirror of sv_verify_plan in include/specverify.h."""
    _fields_ = [
        ("grouped", ctypes.c_int),
        ("clusters", ctypes.c_int),
        ("cluster_size", ctypes.c_int),
        ("max_seqs_per_cluster", ctypes.c_int),
    ]


_lock = threading.Lock()
_lib = None

# (name, restype, argtypes) of every symbol the header declares.
P = ctypes.c_void_p
I = ctypes.c_int
SIGNATURES = [
    ("spec_verify", I, [P, P, P, I, I, I, I, ctypes.c_float, I, ctypes.c_uint64, P, P, P]),
    ("spec_verify_ex", I, [ctypes.POINTER(sv_verify_args)]),
    ("spec_verify_plan", I, [ctypes.POINTER(sv_verify_args), ctypes.POINTER(sv_verify_plan)]),
    ("spec_verify_lmhead_workspace_bytes", ctypes.c_size_t, [I, I, I, I]),
    ("spec_verify_lmhead", I, [P, P, P, P, I, I, I, I, I, ctypes.c_float, I, ctypes.c_uint64, P,
                               ctypes.c_size_t, P, P, P]),
    ("spec_lmhead_logits", I, [P, P, I, I, I, P, P]),
    ("spec_verify_tree", I, [P, I, P, P, I, I, I, P, P, P, P]),
    ("spec_prompt_lookup", I, [P, P, I, I, I, I, P, P, P]),
    ("spec_commit", I, [P, P, I, I, P, P, I, P, P]),
    ("spec_verify_lmhead_noalloc", I, [P, P, P, P, I, I, I, I, I, ctypes.c_float, I,
                                       ctypes.c_uint64, P, P, P]),
    ("sv_status_string", ctypes.c_char_p, [I]),
    ("sv_last_cuda_error", I, []),
    ("sv_version", I, []),
    ("sv_verify_args_size", ctypes.c_size_t, []),
]


def load_library(path: str):
    """Load one build of the library (release or debug) and declare the
    signatures of every symbol the header declares; fail loudly when it has
    not been built."""
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (there is no fallback)")
    lib = ctypes.CDLL(path)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if lib.sv_verify_args_size() != ctypes.sizeof(sv_verify_args):
        raise ImportError("sv_verify_args layout differs between the binding and the library")
    return lib


def _load():
    """The in-tree release library, loaded once."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(LIB_PATH)
    return _lib


def library():
    return _load()


def sv_status_string(status: int) -> str:
    return _load().sv_status_string(int(status)).decode()


def sv_version() -> int:
    return int(_load().sv_version())


def _check(status: int, where: str):
    if status != 0:
        raise SpecVerifyError(int(status), where)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SV_F32
    if t.dtype == torch.bfloat16:
        return SV_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _mode_code(mode) -> int:
    if mode in ("greedy", SV_GREEDY):
        return SV_GREEDY
    if mode in ("sample", SV_SAMPLE):
        return SV_SAMPLE
    raise ValueError(f"mode must be 'greedy' or 'sample', got {mode!r}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("every tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("every tensor must be contiguous")
    return t.data_ptr()


def _stream(stream, device):
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def spec_verify(target_logits, draft_logits, draft_tokens, temperature=1.0, mode="sample", seed=0,
                out_tokens=None, out_n_accepted=None, stream=None):
    """Verify a batch: returns (out_tokens [B, K+1] int32, out_n_accepted [B] int32)."""
    B, K1, V = target_logits.shape
    K = K1 - 1
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty(B, K1, dtype=torch.int32, device=dev)
    if out_n_accepted is None:
        out_n_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        st = _load().spec_verify(
            _ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens), B, K, V,
            _dtype_code(target_logits), float(temperature), _mode_code(mode),
            ctypes.c_uint64(int(seed) & (2**64 - 1)), _ptr(out_tokens), _ptr(out_n_accepted),
            _stream(stream, dev))
    _check(st, "spec_verify")
    return out_tokens, out_n_accepted


def spec_verify_ex(target_logits, draft_logits, draft_tokens, temperature=1.0, modes="sample",
                   seed=0, seq_ids=None, out_tokens=None, out_n_accepted=None, out_p_target=None,
                   out_p_draft=None, out_residual_mass=None, status_word=None, cluster_size=0,
                   stream=None, debug=False, overlap_previous=False, draft_lens=None, flags=0,
                   out_draw_edges=None, lib=None, seqs_per_cluster=0, plan_only=False):
    """Verify with per-sequence modes ([B] int32 tensor, or 'greedy'/'sample'
    for all), explicit Philox sequence ids and optional debug outputs.
    debug=True allocates out_p_target, out_p_draft, out_residual_mass,
    out_draw_edges and status_word. overlap_previous=True sets SV_ARG_OVERLAP_PREVIOUS (the
    inputs are not written by the work just before this call on the stream).
    draft_lens: optional [B] int32 device tensor of per-sequence draft counts.
    lib: a handle from load_library() to call another build of the library
    (the debug build); the release library by default.
    seqs_per_cluster: 0 automatic, 1 one cluster per sequence, 2..8 that many
    sequences per cluster of cluster_size CTAs (calls without overlap).
    plan_only=True: enqueue nothing and return the launch the call would make
    (spec_verify_plan): {"grouped", "clusters", "cluster_size",
    "max_seqs_per_cluster"}.
    Returns a dict of the output tensors."""
    B, K1, V = target_logits.shape
    K = K1 - 1
    dev = target_logits.device
    a = sv_verify_args()
    if out_tokens is None:
        out_tokens = torch.empty(B, K1, dtype=torch.int32, device=dev)
    if out_n_accepted is None:
        out_n_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    if debug:
        if out_p_target is None:
            out_p_target = torch.empty(B, K, dtype=torch.float32, device=dev)
        if out_p_draft is None:
            out_p_draft = torch.empty(B, K, dtype=torch.float32, device=dev)
        if out_residual_mass is None:
            out_residual_mass = torch.empty(B, dtype=torch.float32, device=dev)
        if status_word is None:
            status_word = torch.zeros(1, dtype=torch.int32, device=dev)
        if out_draw_edges is None:
            out_draw_edges = torch.empty(B, 2, dtype=torch.float32, device=dev)
    a.target_logits = _ptr(target_logits)
    a.draft_logits = _ptr(draft_logits)
    a.draft_tokens = _ptr(draft_tokens)
    a.B, a.K, a.V = B, K, V
    a.dtype = _dtype_code(target_logits)
    a.temperature = float(temperature)
    if isinstance(modes, torch.Tensor):
        a.mode = SV_SAMPLE
        a.modes = _ptr(modes)
    else:
        a.mode = _mode_code(modes)
        a.modes = None
    a.seed = int(seed) & (2**64 - 1)
    a.seq_ids = _ptr(seq_ids)
    a.out_tokens = _ptr(out_tokens)
    a.out_n_accepted = _ptr(out_n_accepted)
    a.out_p_target = _ptr(out_p_target)
    a.out_p_draft = _ptr(out_p_draft)
    a.out_residual_mass = _ptr(out_residual_mass)
    a.status_word = _ptr(status_word)
    a.cluster_size = int(cluster_size)
    a.flags = (SV_ARG_OVERLAP_PREVIOUS if overlap_previous else 0) | int(flags)
    a.draft_lens = _ptr(draft_lens)
    a.out_draw_edges = _ptr(out_draw_edges)
    a.seqs_per_cluster = int(seqs_per_cluster)
    with torch.cuda.device(dev):
        a.stream = _stream(stream, dev)
        if plan_only:
            plan = sv_verify_plan()
            st = (lib or _load()).spec_verify_plan(ctypes.byref(a), ctypes.byref(plan))
            _check(st, "spec_verify_plan")
            return {"grouped": bool(plan.grouped), "clusters": plan.clusters, "cluster_size": plan.cluster_size,
                    "max_seqs_per_cluster": plan.max_seqs_per_cluster}
        st = (lib or _load()).spec_verify_ex(ctypes.byref(a))
    _check(st, "spec_verify_ex")
    return {"tokens": out_tokens, "n_accepted": out_n_accepted, "p_target": out_p_target,
            "p_draft": out_p_draft, "residual_mass": out_residual_mass,
            "draw_edges": out_draw_edges, "status_word": status_word}


def spec_verify_plan(target_logits, draft_logits, draft_tokens, temperature=1.0, **kw):
    """The launch spec_verify_ex would make for these arguments (nothing is
    enqueued): {"grouped", "clusters", "cluster_size", "max_seqs_per_cluster"}."""
    return spec_verify_ex(target_logits, draft_logits, draft_tokens, temperature, plan_only=True, **kw)


def spec_verify_tree(target_logits, tree_tokens, tree_parents, out_tokens=None, out_n_accepted=None,
                     out_last_node=None, stream=None):
    """Greedy tree verification: target_logits [B, N, V], tree_tokens and
    tree_parents [B, N] int32 (node 0 is the root). Returns (tokens [B, N],
    n_accepted [B], last_node [B])."""
    B, N, V = target_logits.shape
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty(B, N, dtype=torch.int32, device=dev)
    if out_n_accepted is None:
        out_n_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    if out_last_node is None:
        out_last_node = torch.empty(B, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        st = _load().spec_verify_tree(_ptr(target_logits), _dtype_code(target_logits), _ptr(tree_tokens),
                                      _ptr(tree_parents), B, N, V, _ptr(out_tokens), _ptr(out_n_accepted),
                                      _ptr(out_last_node), _stream(stream, dev))
    _check(st, "spec_verify_tree")
    return out_tokens, out_n_accepted, out_last_node


def spec_prompt_lookup(tokens, lengths, max_ngram=3, n_drafts=5, out_drafts=None, out_n_drafts=None,
                       stream=None):
    """Prompt lookup drafting: tokens [B, L_max] int32, lengths [B] int32
    (device). Returns (drafts [B, n_drafts] -1 padded, n_drafts [B])."""
    B, L_max = tokens.shape
    dev = tokens.device
    if out_drafts is None:
        out_drafts = torch.empty(B, n_drafts, dtype=torch.int32, device=dev)
    if out_n_drafts is None:
        out_n_drafts = torch.empty(B, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        st = _load().spec_prompt_lookup(_ptr(tokens), _ptr(lengths), B, L_max, int(max_ngram),
                                        int(n_drafts), _ptr(out_drafts), _ptr(out_n_drafts),
                                        _stream(stream, dev))
    _check(st, "spec_prompt_lookup")
    return out_drafts, out_n_drafts


def spec_commit(tokens, lengths, out_tokens, n_accepted, out_n_committed=None, stream=None):
    """Append each sequence's accepted drafts and next token to its context
    (tokens [B, L_max], lengths [B], updated in place). Returns the number of
    tokens committed per sequence."""
    B, L_max = tokens.shape
    K = out_tokens.shape[1] - 1
    dev = tokens.device
    if out_n_committed is None:
        out_n_committed = torch.empty(B, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        st = _load().spec_commit(_ptr(tokens), _ptr(lengths), B, L_max, _ptr(out_tokens), _ptr(n_accepted), K,
                                 _ptr(out_n_committed), _stream(stream, dev))
    _check(st, "spec_commit")
    return out_n_committed


def spec_lmhead_logits(hidden, W, out=None, stream=None):
    """fp32 logits [M, V] = hidden [M, d] (bf16) . W [d, V] (bf16) on the tensor cores."""
    hidden = hidden.reshape(-1, hidden.shape[-1])
    M, d = hidden.shape
    V = W.shape[1]
    dev = hidden.device
    if out is None:
        out = torch.empty(M, V, dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        st = _load().spec_lmhead_logits(_ptr(hidden), _ptr(W), M, d, V, _ptr(out), _stream(stream, dev))
    _check(st, "spec_lmhead_logits")
    return out


def spec_verify_lmhead_workspace_bytes(B: int, K: int, d: int, V: int) -> int:
    return int(_load().spec_verify_lmhead_workspace_bytes(B, K, d, V))


def spec_verify_lmhead(hidden, W, draft_logits, draft_tokens, temperature=1.0, mode="sample",
                       seed=0, workspace=None, out_tokens=None, out_n_accepted=None, stream=None,
                       lib=None):
    """Fused LM head + verify: hidden [B, K+1, d] bf16, W [d, V] bf16. lib: as
    in spec_verify_ex."""
    B, K1, d = hidden.shape
    K = K1 - 1
    V = W.shape[1]
    dev = hidden.device
    need = spec_verify_lmhead_workspace_bytes(B, K, d, V)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty(B, K1, dtype=torch.int32, device=dev)
    if out_n_accepted is None:
        out_n_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    ddt = _dtype_code(draft_logits) if draft_logits is not None else SV_BF16
    with torch.cuda.device(dev):
        st = (lib or _load()).spec_verify_lmhead(
            _ptr(hidden), _ptr(W), _ptr(draft_logits), _ptr(draft_tokens), B, K, d, V, ddt,
            float(temperature), _mode_code(mode), ctypes.c_uint64(int(seed) & (2**64 - 1)),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out_tokens),
            _ptr(out_n_accepted), _stream(stream, dev))
    _check(st, "spec_verify_lmhead")
    return out_tokens, out_n_accepted


def spec_verify_lmhead_noalloc(hidden, W, draft_logits, draft_tokens, temperature=1.0,
                               mode="sample", seed=0, out_tokens=None, out_n_accepted=None,
                               stream=None):
    """spec_verify_lmhead with its workspace (logits and per-tile partials)
    in the library's own static device scratch (SV_LMHEAD_SCRATCH_BYTES): the
    C call allocates nothing. Calls
    that may overlap on one device race on that scratch; order them."""
    B, K1, d = hidden.shape
    K = K1 - 1
    V = W.shape[1]
    dev = hidden.device
    if out_tokens is None:
        out_tokens = torch.empty(B, K1, dtype=torch.int32, device=dev)
    if out_n_accepted is None:
        out_n_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    ddt = _dtype_code(draft_logits) if draft_logits is not None else SV_BF16
    with torch.cuda.device(dev):
        st = _load().spec_verify_lmhead_noalloc(
            _ptr(hidden), _ptr(W), _ptr(draft_logits), _ptr(draft_tokens), B, K, d, V, ddt,
            float(temperature), _mode_code(mode), ctypes.c_uint64(int(seed) & (2**64 - 1)),
            _ptr(out_tokens), _ptr(out_n_accepted), _stream(stream, dev))
    _check(st, "spec_verify_lmhead_noalloc")
    return out_tokens, out_n_accepted
