"""The C ABI without a GPU: the library loads, exports every function the
headers declare, and rejects bad arguments on the host before any CUDA call
(so these run on a machine with no driver)."""

import ctypes
import os
import re

import pytest

import exact_attention_90_gb300 as fa
from exact_attention_90_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return fa.load_library()


def declared_functions():
    names = set()
    for h in os.listdir(INCLUDE):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(INCLUDE, h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(fa_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_headers_declare_the_abi():
    names = declared_functions()
    for n in ("fa_fwd", "fa_status_string", "fa_version", "fa_debug_sync_check",
              "fa_last_cuda_error", "fa_unit_tma", "fa_unit_qk", "fa_unit_pv", "fa_unit_timeout",
              "fa_fwd_simt", "fa_fwd_split", "fa_fwd_split_workspace_size", "fa_fwd_window",
              "fa_fwd_split_heuristic", "fa_bwd", "fa_bwd_workspace_size"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"libfa.so does not export {n}"
    # and the binding wraps each of them under the same name
    wrapped = {name for name, _, _ in fa.EXPORTS}
    assert set(declared_functions()) <= wrapped
    for n in declared_functions():
        assert callable(getattr(fa, n))


def test_version_and_status_strings(lib):
    assert fa.fa_version() == 10000
    for s in range(7):
        txt = fa.fa_status_string(s)
        assert isinstance(txt, str) and txt
    assert fa.fa_status_string(0) == "ok"
    assert fa.fa_status_string(99) == "unknown status"


# fake, 16-byte aligned, far-apart device addresses: validation never touches them
BASE = 1 << 44
Q, K, V, O, L = (BASE + (i << 36) for i in range(5))
GOOD = dict(q=Q, k=K, v=V, o=O, lse=L, B=2, Hq=4, Hkv=2, T=100, d=64, scale=0.125, causal=1,
            dtype=fa.FA_DTYPE_BF16)


def call(**kw):
    a = dict(GOOD)
    a.update(kw)
    return fa.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"],
                     a["T"], a["d"], a["scale"], a["causal"], a["dtype"], stream=0)


@pytest.mark.parametrize("kw,status", [
    (dict(q=0), fa.FA_ERR_INVALID_ARG),
    (dict(k=0), fa.FA_ERR_INVALID_ARG),
    (dict(v=0), fa.FA_ERR_INVALID_ARG),
    (dict(o=0), fa.FA_ERR_INVALID_ARG),
    (dict(lse=0), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(Hq=-1), fa.FA_ERR_INVALID_ARG),
    (dict(Hkv=0), fa.FA_ERR_INVALID_ARG),
    (dict(T=0), fa.FA_ERR_INVALID_ARG),
    (dict(d=0), fa.FA_ERR_INVALID_ARG),
    (dict(Hq=4, Hkv=3), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(causal=2), fa.FA_ERR_INVALID_ARG),
    (dict(d=48), fa.FA_ERR_UNSUPPORTED),
    (dict(d=256), fa.FA_ERR_UNSUPPORTED),
    (dict(dtype=7), fa.FA_ERR_UNSUPPORTED),
    (dict(q=Q + 8), fa.FA_ERR_MISALIGNED),
    (dict(o=O + 4), fa.FA_ERR_MISALIGNED),
    (dict(lse=L + 2), fa.FA_ERR_MISALIGNED),
    (dict(o=Q), fa.FA_ERR_INVALID_ARG),          # output aliases an input
    (dict(o=K + 4096), fa.FA_ERR_INVALID_ARG),   # output overlaps K
    (dict(lse=O + 64), fa.FA_ERR_INVALID_ARG),   # the two outputs overlap
    (dict(B=1 << 20, Hq=1 << 12, Hkv=1 << 12, T=1 << 20), fa.FA_ERR_INVALID_ARG),  # size overflow
    (dict(B=1, Hq=1, Hkv=1, T=1 << 30), fa.FA_ERR_INVALID_ARG),  # T >= 2^30
])
def test_fwd_rejects_bad_arguments_on_the_host(lib, kw, status):
    assert call(**kw) == status
    # same checks for the CUDA-core entry point
    a = dict(GOOD)
    a.update(kw)
    assert fa.fa_fwd_simt(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"],
                          a["T"], a["d"], a["scale"], a["causal"], a["dtype"], stream=0) == status


def test_unit_entry_points_reject_bad_arguments(lib):
    assert fa.fa_unit_tma(0, O, 64, stream=0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_unit_tma(Q, O, 48, stream=0) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_unit_tma(Q + 4, O, 64, stream=0) == fa.FA_ERR_MISALIGNED
    assert fa.fa_unit_qk(Q, 0, O, 64, stream=0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_unit_qk(Q, K, O, 8, stream=0) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_unit_pv(Q, 0, K, 0, 64, stream=0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_unit_pv(Q, 0, K, O, 64, mode=4, stream=0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_unit_pv(0, 0, K, O, 64, mode=0, stream=0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_unit_pv(Q, 0, K, O, 64, mode=2, stream=0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_unit_pv(Q, 0, K, O, 64, lbo=8, stream=0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_unit_timeout(1000, 0, stream=0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_unit_timeout(0, O, stream=0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_unit_timeout(1 << 40, O, stream=0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_unit_timeout(1000, O + 2, stream=0) == fa.FA_ERR_MISALIGNED
    # the pipe-rate probe: kind 0..2, iterations 1..2^24, blocks 1..4096, both pointers
    assert fa.fa_unit_pipe_rate(0, 16, 152, 0, O, stream=0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_unit_pipe_rate(0, 16, 152, O, 0, stream=0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_unit_pipe_rate(3, 16, 152, O, O, stream=0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_unit_pipe_rate(0, 0, 152, O, O, stream=0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_unit_pipe_rate(0, (1 << 24) + 1, 152, O, O, stream=0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_unit_pipe_rate(0, 16, 0, O, O, stream=0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_unit_pipe_rate(0, 16, 4097, O, O, stream=0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_unit_pipe_rate(0, 16, 152, O + 2, O, stream=0) == fa.FA_ERR_MISALIGNED
    assert fa.fa_unit_pipe_rate(0, 16, 152, O, O + 4, stream=0) == fa.FA_ERR_MISALIGNED


def test_tensor_api_refuses_cpu_tensors():
    import torch

    q = torch.zeros(1, 1, 8, 16)
    with pytest.raises(TypeError):
        fa.fwd(q, q, q)


def test_exported_symbols_have_c_linkage(lib):
    # a C++-mangled name would not be found by its plain name
    for n in declared_functions():
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


WS = BASE + (6 << 36)


def split_call(num_splits=4, ws=WS, ws_bytes=None, **kw):
    a = dict(GOOD)
    a.update(kw)
    if ws_bytes is None:
        ws_bytes = fa.fa_fwd_split_workspace_size(a["B"], a["Hq"], a["T"], a["d"], num_splits)
    return fa.fa_fwd_split(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"],
                           a["T"], a["d"], a["scale"], a["causal"], a["dtype"], num_splits, ws,
                           ws_bytes, stream=0)


def test_split_workspace_size_and_heuristic(lib):
    # num_splits * B * Hq * T * (d + 1) * 4 bytes
    assert fa.fa_fwd_split_workspace_size(2, 4, 100, 64, 3) == 3 * 2 * 4 * 100 * 65 * 4
    assert fa.fa_fwd_split_workspace_size(2, 4, 100, 64, 0) == 0
    assert fa.fa_fwd_split_workspace_size(2, 4, 100, 64, 65) == 0
    assert fa.fa_fwd_split_workspace_size(0, 4, 100, 64, 2) == 0
    # many row blocks: no split; a single small head: split, at most one per KV tile
    assert fa.fa_fwd_split_heuristic(64, 1, 1, 4096, 128, 1) == 1
    s = fa.fa_fwd_split_heuristic(1, 1, 1, 4096, 128, 1)
    assert 2 <= s <= 8                                          # >= 4 of the 32 KV tiles each
    assert fa.fa_fwd_split_heuristic(1, 1, 1, 1024, 64, 0) == 2
    assert fa.fa_fwd_split_heuristic(1, 1, 1, 200, 64, 0) == 1  # too short to split
    assert fa.fa_fwd_split_heuristic(0, 1, 1, 200, 64, 0) == 1


def test_split_rejects_bad_arguments_on_the_host(lib):
    assert split_call(num_splits=0) == fa.FA_ERR_INVALID_ARG
    assert split_call(num_splits=65) == fa.FA_ERR_INVALID_ARG
    assert split_call(ws=0) == fa.FA_ERR_WORKSPACE
    assert split_call(ws_bytes=1000) == fa.FA_ERR_WORKSPACE
    assert split_call(ws=WS + 8) == fa.FA_ERR_MISALIGNED
    assert split_call(ws=O) == fa.FA_ERR_INVALID_ARG        # workspace overlaps O
    assert split_call(q=0) == fa.FA_ERR_INVALID_ARG         # the fa_fwd checks apply too
    assert split_call(d=48) == fa.FA_ERR_UNSUPPORTED


def test_window_rejects_bad_arguments_on_the_host(lib):
    a = dict(GOOD)

    def wcall(wl, wr, **kw):
        b = dict(a)
        b.update(kw)
        return fa.fa_fwd_window(b["q"], b["k"], b["v"], b["o"], b["lse"], b["B"], b["Hq"],
                                b["Hkv"], b["T"], b["d"], b["scale"], wl, wr, b["dtype"], stream=0)

    assert wcall(-2, 4) == fa.FA_ERR_INVALID_ARG
    assert wcall(4, -5) == fa.FA_ERR_INVALID_ARG
    assert wcall(4, 4, q=0) == fa.FA_ERR_INVALID_ARG
    assert wcall(4, 4, d=24) == fa.FA_ERR_UNSUPPORTED
    assert wcall(4, 4, o=O + 2) == fa.FA_ERR_MISALIGNED


DO, DQ, DK, DV, BWS = (BASE + ((7 + i) << 36) for i in range(5))


def bwd_call(ws_bytes=None, **kw):
    a = dict(GOOD, d_o=DO, dq=DQ, dk=DK, dv=DV, ws=BWS, wl=-1, wr=-1)
    a.update(kw)
    if ws_bytes is None:
        ws_bytes = fa.fa_bwd_workspace_size(a["B"], a["Hq"], a["T"])
    return fa.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["d_o"], a["dq"], a["dk"],
                     a["dv"], a["B"], a["Hq"], a["Hkv"], a["T"], a["d"], a["scale"], a["causal"],
                     a["wl"], a["wr"], a["dtype"], a["ws"], ws_bytes, stream=0)


def test_bwd_workspace_size(lib):
    # two fp32 values per query row, rows padded to a multiple of 128 per head
    assert fa.fa_bwd_workspace_size(2, 4, 100) == 2 * 2 * 4 * 128 * 4
    assert fa.fa_bwd_workspace_size(1, 1, 128) == 2 * 128 * 4
    assert fa.fa_bwd_workspace_size(1, 1, 129) == 2 * 256 * 4
    assert fa.fa_bwd_workspace_size(0, 1, 10) == 0
    assert fa.fa_bwd_workspace_size(1, 1, 0) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(q=0), fa.FA_ERR_INVALID_ARG),            # the forward's checks apply
    (dict(o=0), fa.FA_ERR_INVALID_ARG),
    (dict(lse=0), fa.FA_ERR_INVALID_ARG),
    (dict(d_o=0), fa.FA_ERR_INVALID_ARG),
    (dict(dq=0), fa.FA_ERR_INVALID_ARG),
    (dict(dk=0), fa.FA_ERR_INVALID_ARG),
    (dict(dv=0), fa.FA_ERR_INVALID_ARG),
    (dict(d=48), fa.FA_ERR_UNSUPPORTED),
    (dict(Hq=4, Hkv=3), fa.FA_ERR_INVALID_ARG),
    (dict(wl=-2), fa.FA_ERR_INVALID_ARG),
    (dict(wr=-3), fa.FA_ERR_INVALID_ARG),
    (dict(d_o=DO + 8), fa.FA_ERR_MISALIGNED),
    (dict(dk=DK + 2), fa.FA_ERR_MISALIGNED),
    (dict(ws=0), fa.FA_ERR_WORKSPACE),
    (dict(ws_bytes=100), fa.FA_ERR_WORKSPACE),
    (dict(ws=BWS + 4), fa.FA_ERR_MISALIGNED),
    (dict(dq=Q), fa.FA_ERR_INVALID_ARG),           # a gradient aliases an input
    (dict(dk=DO + 4096), fa.FA_ERR_INVALID_ARG),   # dK overlaps dO
    (dict(dv=DK), fa.FA_ERR_INVALID_ARG),          # two gradients alias
    (dict(ws=DQ + 64), fa.FA_ERR_INVALID_ARG),     # the workspace overlaps dQ
    (dict(ws=O), fa.FA_ERR_INVALID_ARG),           # the workspace overlaps O
])
def test_bwd_rejects_bad_arguments_on_the_host(lib, kw, status):
    assert bwd_call(**kw) == status


def test_bwd_tensor_api_refuses_cpu_tensors():
    import torch

    q = torch.zeros(1, 1, 8, 16)
    lse = torch.zeros(1, 1, 8)
    with pytest.raises(TypeError):
        fa.bwd(q, q, q, q, lse, q)


GT, LWS = BASE + (12 << 36), BASE + (13 << 36)


def lg_call(w=3, gt=GT, n=5, ws=LWS, ws_bytes=None, **kw):
    a = dict(GOOD)
    a.update(kw)
    if ws_bytes is None:
        ws_bytes = fa.fa_fwd_local_global_workspace_size(a["T"])
    return fa.fa_fwd_local_global(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"],
                                  a["Hkv"], a["T"], a["d"], a["scale"], a["causal"], w, gt, n,
                                  a["dtype"], ws, ws_bytes, stream=0)


def test_local_global_workspace_size(lib):
    # 16 bytes of key bits and 4 bytes of tile list per 128-key tile, plus 16
    assert fa.fa_fwd_local_global_workspace_size(128) == 48
    assert fa.fa_fwd_local_global_workspace_size(1000) == 8 * 20 + 16
    assert fa.fa_fwd_local_global_workspace_size(0) == 0


def test_local_global_packed_workspace_size(lib):
    # the tile-mode bytes, then R ints (R = tokens rounded up to 128, at least
    # 128), a 16-byte count and the packed K and V rows: 2 * B * Hkv * R * d * 2
    lg = fa.fa_fwd_local_global_workspace_size(1000)
    bf16, f32 = fa.FA_DTYPE_BF16, fa.FA_DTYPE_F32
    assert (fa.fa_fwd_local_global_packed_workspace_size(2, 4, 1000, 64, bf16, 37)
            == lg + 128 * 4 + 16 + 2 * 2 * 4 * 128 * 64 * 2)
    assert (fa.fa_fwd_local_global_packed_workspace_size(1, 1, 1000, 128, bf16, 300)
            == lg + 384 * 4 + 16 + 2 * 384 * 128 * 2)
    # fp32 inputs and no tokens need no packing; invalid sizes give 0
    assert fa.fa_fwd_local_global_packed_workspace_size(2, 4, 1000, 64, f32, 37) == lg
    assert fa.fa_fwd_local_global_packed_workspace_size(2, 4, 1000, 64, bf16, 0) == lg
    assert fa.fa_fwd_local_global_packed_workspace_size(0, 4, 1000, 64, bf16, 3) == 0
    assert fa.fa_fwd_local_global_packed_workspace_size(2, 4, 1000, 64, bf16, -1) == 0
    assert fa.fa_fwd_local_global_packed_workspace_size(2, 4, 1000, 64, 9, 3) == 0


def test_local_global_rejects_bad_arguments_on_the_host(lib):
    assert lg_call(w=-1) == fa.FA_ERR_INVALID_ARG
    assert lg_call(n=-2) == fa.FA_ERR_INVALID_ARG
    assert lg_call(gt=0, n=3) == fa.FA_ERR_INVALID_ARG
    assert lg_call(gt=GT + 2) == fa.FA_ERR_MISALIGNED
    assert lg_call(ws=0) == fa.FA_ERR_WORKSPACE
    assert lg_call(ws_bytes=16) == fa.FA_ERR_WORKSPACE
    assert lg_call(ws=LWS + 8) == fa.FA_ERR_MISALIGNED
    assert lg_call(ws=O) == fa.FA_ERR_INVALID_ARG            # workspace overlaps O
    assert lg_call(gt=O + 64) == fa.FA_ERR_INVALID_ARG       # tokens overlap an output
    assert lg_call(q=0) == fa.FA_ERR_INVALID_ARG             # the fa_fwd checks apply
    assert lg_call(d=40) == fa.FA_ERR_UNSUPPORTED
    # with the packing size the overlap check covers the packed K/V rows too:
    # a workspace that ends 64 bytes before O in whole-tile mode reaches into
    # O once it is large enough to pack
    lg = fa.fa_fwd_local_global_workspace_size(GOOD["T"])
    packed = fa.fa_fwd_local_global_packed_workspace_size(GOOD["B"], GOOD["Hkv"], GOOD["T"],
                                                          GOOD["d"], GOOD["dtype"], 5)
    assert packed > lg + 64
    assert lg_call(ws=O - lg - 64, ws_bytes=packed) == fa.FA_ERR_INVALID_ARG


def test_bwd_local_global_workspace_and_host_errors(lib):
    assert (fa.fa_bwd_local_global_workspace_size(2, 4, 100)
            == fa.fa_bwd_workspace_size(2, 4, 100) + fa.fa_fwd_local_global_workspace_size(100))
    assert fa.fa_bwd_local_global_workspace_size(0, 4, 100) == 0
    need = fa.fa_bwd_local_global_workspace_size(GOOD["B"], GOOD["Hq"], GOOD["T"])

    def call(w=3, gt=GT, n=5, ws=BWS, ws_bytes=need, **kw):
        a = dict(GOOD, d_o=DO, dq=DQ, dk=DK, dv=DV)
        a.update(kw)
        return fa.fa_bwd_local_global(a["q"], a["k"], a["v"], a["o"], a["lse"], a["d_o"], a["dq"],
                                      a["dk"], a["dv"], a["B"], a["Hq"], a["Hkv"], a["T"], a["d"],
                                      a["scale"], a["causal"], w, gt, n, a["dtype"], ws, ws_bytes,
                                      stream=0)

    assert call(w=-1) == fa.FA_ERR_INVALID_ARG
    assert call(n=-1) == fa.FA_ERR_INVALID_ARG
    assert call(gt=0, n=2) == fa.FA_ERR_INVALID_ARG
    assert call(gt=GT + 2) == fa.FA_ERR_MISALIGNED
    assert call(ws_bytes=need - 16) == fa.FA_ERR_WORKSPACE      # the key sets do not fit
    assert call(dq=GT) == fa.FA_ERR_INVALID_ARG                  # dQ overlaps the token list
    assert call(dq=0) == fa.FA_ERR_INVALID_ARG                   # the fa_bwd checks apply
    assert call(d=24) == fa.FA_ERR_UNSUPPORTED
