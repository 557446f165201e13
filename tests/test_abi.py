"""The C ABI library loads, exports every symbol include/*.h declares, and
rejects bad arguments on the host (CPU only: no call here reaches the GPU)."""
import ctypes
import glob
import os
import re

import pytest

from speculative_decoding_verification_24_gb300 import binding
from speculative_decoding_verification_24_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return binding.library()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b([A-Za-z_][A-Za-z0-9_]*)\s*\(", text):
            name = m.group(1)
            # a function declaration: identifier followed by '(' at file scope
            line_start = text.rfind("\n", 0, m.start()) + 1
            prefix = text[line_start:m.start()]
            if name in {"defined", "if", "sizeof"} or prefix.strip().startswith("#"):
                continue
            if re.search(r"[;{}]\s*$", prefix) or prefix.strip() == "":
                continue
            names.add(name)
    return names


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("spec_verify", "spec_verify_ex", "spec_verify_lmhead",
                     "spec_verify_lmhead_workspace_bytes", "sv_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names
    so = ctypes.CDLL(binding.LIB_PATH)
    for name in sorted(names):
        assert hasattr(so, name), f"{name} declared but not exported"
    bound = {n for n, _, _ in binding.SIGNATURES}
    assert names <= bound, f"binding misses {sorted(names - bound)}"


def test_debug_build_exports_the_same_boundary(lib):
    # libspecverify_debug.so: the same sources with SPECVERIFY_DEBUG (bounds
    # checks in the verify kernel); it loads without a GPU like the release
    # build and exports every declared symbol with the same struct layout
    dbg = binding.load_library(binding.DEBUG_LIB_PATH)
    so = ctypes.CDLL(binding.DEBUG_LIB_PATH)
    for name in sorted(declared_functions()):
        assert hasattr(so, name), f"{name} declared but not exported by the debug build"
    assert dbg.sv_verify_args_size() == ctypes.sizeof(binding.sv_verify_args)
    assert dbg.sv_version() == lib.sv_version()
    # host validation is the same code in both builds
    assert dbg.spec_verify_lmhead_workspace_bytes(32, 5, 4096, 128256) == \
        lib.spec_verify_lmhead_workspace_bytes(32, 5, 4096, 128256)


def test_struct_layout_matches(lib):
    assert lib.sv_verify_args_size() == ctypes.sizeof(binding.sv_verify_args)
    assert lib.sv_version() >= 100
    assert lib.sv_status_string(0).decode() == "ok"
    for code in range(13):
        assert lib.sv_status_string(code)


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def call(lib, target=FAKE, draft=FAKE, tokens=FAKE, B=2, K=4, V=100, dtype=0, T=1.0, mode=1,
         out_tokens=FAKE, out_n=FAKE):
    return lib.spec_verify(target, draft, tokens, B, K, V, dtype, T, mode, 0, out_tokens, out_n,
                           None)


@pytest.mark.parametrize("kwargs,code", [
    (dict(target=None), 1), (dict(tokens=None), 1), (dict(out_tokens=None), 1),
    (dict(out_n=None), 1), (dict(draft=None, mode=1), 1),
    (dict(B=0), 2), (dict(K=0), 2), (dict(K=32), 2), (dict(V=1), 2),
    (dict(dtype=7), 3),
    (dict(T=0.0), 4), (dict(T=-1.0), 4), (dict(T=float("nan")), 4), (dict(T=float("inf")), 4),
    (dict(T=1e-40), 4),
    (dict(mode=5), 8),
    (dict(target=FAKE + 2, dtype=0), 9), (dict(draft=FAKE + 1, dtype=1), 9),
    (dict(tokens=FAKE + 2), 9),
])
def test_host_validation(lib, kwargs, code):
    assert call(lib, **kwargs) == code


def test_greedy_ignores_temperature_and_draft_validation_order(lib):
    # greedy with a NULL draft and a bad temperature is valid up to the device
    # check; here a bad shape still comes first
    assert call(lib, draft=None, mode=0, T=float("nan"), B=0) == 2


def test_ex_validation(lib):
    a = binding.sv_verify_args()
    assert lib.spec_verify_ex(None) == 1
    assert lib.spec_verify_ex(ctypes.byref(a)) == 1
    a.target_logits = a.draft_logits = a.draft_tokens = a.out_tokens = a.out_n_accepted = FAKE
    a.B, a.K, a.V, a.dtype, a.temperature, a.mode = 2, 3, 64, 0, 1.0, 1
    a.cluster_size = 3
    assert lib.spec_verify_ex(ctypes.byref(a)) == 10
    a.cluster_size = 32
    assert lib.spec_verify_ex(ctypes.byref(a)) == 10
    a.cluster_size = 0
    a.seq_ids = FAKE + 4
    assert lib.spec_verify_ex(ctypes.byref(a)) == 9


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(ImportError):
        binding.library()


def test_lmhead_workspace_size(lib):
    # fp32 logits of B * (K+1) rows, then one 8-byte partial per target row
    # and 128-column tile, then one per draft row and tile, each rounded up
    # to 256 bytes
    assert (lib.spec_verify_lmhead_workspace_bytes(32, 5, 4096, 128256)
            == 32 * 6 * 128256 * 4 + 1002 * 192 * 8 + 1002 * 160 * 8)
    assert lib.spec_verify_lmhead_workspace_bytes(1, 1, 64, 8) == 256 + 256 + 256
    assert lib.spec_verify_lmhead_workspace_bytes(3, 4, 64, 1000) == 60160 + 1024 + 768
    assert lib.spec_verify_lmhead_workspace_bytes(0, 1, 64, 8) == 0


def lm_call(lib, hidden=FAKE, W=FAKE, draft=FAKE, tokens=FAKE, B=2, K=3, d=128, V=256, ddt=1,
            T=1.0, mode=1, ws=FAKE, ws_bytes=1 << 30, out_tokens=FAKE, out_n=FAKE):
    return lib.spec_verify_lmhead(hidden, W, draft, tokens, B, K, d, V, ddt, T, mode, 0, ws,
                                  ws_bytes, out_tokens, out_n, None)


@pytest.mark.parametrize("kwargs,code", [
    (dict(hidden=None), 1), (dict(W=None), 1), (dict(tokens=None), 1), (dict(out_n=None), 1),
    (dict(draft=None, mode=1), 1),
    (dict(B=0), 2), (dict(K=32), 2), (dict(d=100), 2), (dict(d=0), 2), (dict(V=100), 2),
    (dict(B=64, K=4), 2),  # 256 rows fit, 320 do not
    (dict(ddt=4), 3), (dict(T=0.0), 4), (dict(mode=3), 8),
    (dict(ws=None), 5), (dict(ws_bytes=1000), 5),
    (dict(hidden=FAKE + 8), 9), (dict(W=FAKE + 2), 9), (dict(ws=FAKE + 16), 9),
])
def test_lmhead_host_validation(lib, kwargs, code):
    assert lm_call(lib, **kwargs) == code


@pytest.mark.parametrize("args,code", [
    ((None, FAKE, 4, 64, 8, FAKE), 1), ((FAKE, FAKE, 4, 64, 8, None), 1),
    ((FAKE, FAKE, 0, 64, 8, FAKE), 2), ((FAKE, FAKE, 257, 64, 8, FAKE), 2),
    ((FAKE, FAKE, 4, 96, 8, FAKE), 2), ((FAKE, FAKE, 4, 64, 12, FAKE), 2),
    ((FAKE + 4, FAKE, 4, 64, 8, FAKE), 9), ((FAKE, FAKE, 4, 64, 8, FAKE + 2), 9),
])
def test_lmhead_logits_host_validation(lib, args, code):
    assert lib.spec_lmhead_logits(*args, None) == code


@pytest.mark.parametrize("args,code", [
    (dict(target=None), 1), (dict(tokens=None), 1), (dict(parents=None), 1), (dict(out_n=None), 1),
    (dict(B=0), 2), (dict(N=0), 2), (dict(N=33), 2), (dict(V=1), 2), (dict(dtype=5), 3),
    (dict(target=FAKE + 2), 9), (dict(parents=FAKE + 1), 9), (dict(last=FAKE + 2), 9),
])
def test_tree_host_validation(lib, args, code):
    a = dict(target=FAKE, dtype=0, tokens=FAKE, parents=FAKE, B=2, N=8, V=100, out_t=FAKE,
             out_n=FAKE, last=None)
    a.update(args)
    assert lib.spec_verify_tree(a["target"], a["dtype"], a["tokens"], a["parents"], a["B"], a["N"],
                                a["V"], a["out_t"], a["out_n"], a["last"], None) == code


@pytest.mark.parametrize("args,code", [
    (dict(tokens=None), 1), (dict(lengths=None), 1), (dict(out_d=None), 1), (dict(out_n=None), 1),
    (dict(B=0), 2), (dict(L=0), 2), (dict(m=0), 2), (dict(m=17), 2), (dict(k=0), 2), (dict(k=65), 2),
    (dict(tokens=FAKE + 2), 9), (dict(out_n=FAKE + 1), 9),
])
def test_prompt_lookup_host_validation(lib, args, code):
    a = dict(tokens=FAKE, lengths=FAKE, B=2, L=64, m=3, k=5, out_d=FAKE, out_n=FAKE)
    a.update(args)
    assert lib.spec_prompt_lookup(a["tokens"], a["lengths"], a["B"], a["L"], a["m"], a["k"], a["out_d"],
                                  a["out_n"], None) == code


@pytest.mark.parametrize("args,code", [
    (dict(tokens=None), 1), (dict(lengths=None), 1), (dict(out_t=None), 1), (dict(n=None), 1),
    (dict(B=0), 2), (dict(L=0), 2), (dict(K=-1), 2), (dict(K=32), 2),
    (dict(tokens=FAKE + 2), 9), (dict(committed=FAKE + 1), 9),
])
def test_commit_host_validation(lib, args, code):
    a = dict(tokens=FAKE, lengths=FAKE, B=2, L=64, out_t=FAKE, n=FAKE, K=4, committed=None)
    a.update(args)
    assert lib.spec_commit(a["tokens"], a["lengths"], a["B"], a["L"], a["out_t"], a["n"], a["K"],
                           a["committed"], None) == code
