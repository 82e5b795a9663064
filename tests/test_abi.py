"""The C ABI without a GPU: the library loads, exports every function that
include/dit_attn.h declares, and rejects bad arguments on the host (no call
here reaches a kernel; the pointers below are never dereferenced)."""
import ctypes
import os
import re

import pytest
import torch

from sequence_attention_attn_b300 import build, dit_attn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dit_attn.h")

OK, INVALID, SHAPE, MISALIGNED = 0, -1, -2, -3

# Fake, 16-byte aligned device addresses, far apart so that no range overlaps.
A = 0x7F0000000000
B_ = 0x7F1000000000
C = 0x7F2000000000
O = 0x7F3000000000
L = 0x7F4000000000


@pytest.fixture(scope="module")
def lib():
    build.build()
    return dit_attn.lib()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)) - {"defined"})


def test_header_declares_the_boundary():
    names = header_functions()
    for want in ("dit_attn_fwd", "dit_attn_fwd_partials", "dit_attn_merge", "cfg_combine",
                 "cfg_combine_relmae", "dit_attn_fwd_range", "dit_attn_fwd_torus", "dit_last_device_status", "dit_status_string", "dit_abi_version"):
        assert want in names


def test_library_exports_every_header_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), f"{name} declared in dit_attn.h but not exported"
    assert set(header_functions()) <= set(dit_attn.SIGNATURES)


def test_status_strings(lib):
    assert lib.dit_abi_version() == 2
    for code in range(-7, 1):
        s = dit_attn.status_string(code)
        assert s and s != "unknown status"
    assert dit_attn.status_string(-99) == "unknown status"


def fwd(lib, q=A, k=B_, v=C, out=O, lse=L, B=1, H=2, S=256, D=64, n=1):
    return lib.dit_attn_fwd(q, k, v, out, lse, B, H, S, D, n, None)


def test_fwd_rejects_bad_arguments_on_host(lib):
    assert fwd(lib, q=None) == INVALID
    assert fwd(lib, out=None) == INVALID
    assert fwd(lib, B=0) == INVALID
    assert fwd(lib, H=-1) == INVALID
    assert fwd(lib, S=0) == INVALID
    assert fwd(lib, n=0) == INVALID
    assert fwd(lib, n=257) == INVALID            # more chunks than keys
    assert fwd(lib, D=65) == SHAPE
    assert fwd(lib, D=96) == SHAPE
    assert fwd(lib, q=A + 8) == MISALIGNED
    assert fwd(lib, out=O + 4) == MISALIGNED
    assert fwd(lib, lse=L + 2) == MISALIGNED
    assert fwd(lib, out=A + 1024) == INVALID      # out overlaps q
    assert fwd(lib, lse=O + 16) == INVALID        # lse overlaps out


def test_partials_rejects_bad_arguments_on_host(lib):
    f = lib.dit_attn_fwd_partials
    assert f(A, B_, C, None, L, 1, 2, 256, 64, 2, None) == INVALID
    assert f(A, B_, C, O, L + 4, 1, 2, 256, 64, 2, None) == MISALIGNED
    assert f(A, B_, C, O, L, 1, 2, 256, 72, 300, None) == INVALID
    assert f(A, B_, C, A, L, 1, 2, 256, 64, 2, None) == INVALID   # partials overlap q


def test_merge_rejects_bad_arguments_on_host(lib):
    f = lib.dit_attn_merge
    assert f(None, B_, 2, O, L, 100, 64, None) == INVALID
    assert f(A, B_, 0, O, L, 100, 64, None) == INVALID
    assert f(A, B_, 2, O, L, 0, 64, None) == INVALID
    assert f(A, B_, 2, O, L, 100, 0, None) == INVALID
    assert f(A + 4, B_, 2, O, L, 100, 64, None) == MISALIGNED
    assert f(A, B_, 2, A + 64, L, 100, 64, None) == INVALID        # out overlaps partials


def test_cfg_rejects_bad_arguments_on_host(lib):
    f = lib.cfg_combine
    assert f(None, B_, 4.5, O, 100, None) == INVALID
    assert f(A, B_, 4.5, O, 0, None) == INVALID
    assert f(A, B_, float("nan"), O, 100, None) == INVALID
    assert f(A, B_ + 4, 4.5, O, 100, None) == MISALIGNED
    assert f(A, B_, 4.5, A + 16, 100, None) == INVALID             # partial overlap


def test_cfg_relmae_rejects_bad_arguments_on_host(lib):
    f = lib.cfg_combine_relmae
    S_ = 0x7F5000000000
    assert f(A, B_, 4.5, O, 100, None, None) == INVALID             # no sums buffer
    assert f(None, B_, 4.5, O, 100, S_, None) == INVALID
    assert f(A, B_, 4.5, O, 0, S_, None) == INVALID
    assert f(A, B_, float("inf"), O, 100, S_, None) == INVALID
    assert f(A, B_, 4.5, O, 100, S_ + 4, None) == MISALIGNED        # sums not 8-byte aligned
    assert f(A, B_, 4.5, O, 100, A + 64, None) == INVALID           # sums inside eps_c
    assert f(A, B_, 4.5, O, 100, O - 16, None) == INVALID           # sums[2] (the ratio) over out
    assert f(A, B_, 4.5, A + 16, 100, S_, None) == INVALID          # out partly over eps_c


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU behaviour")
def test_valid_call_without_gpu_reports_an_error_not_a_result(lib):
    # Arguments pass the host checks, so the library must reach the CUDA
    # runtime, find no usable device and say so (no CPU fallback).
    rc = fwd(lib)
    assert rc in (-4, -7), rc


def test_python_binding_refuses_cpu_tensors(lib):
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        dit_attn.attention(q, q, q)
    with pytest.raises(ValueError, match="CUDA"):
        dit_attn.combine(torch.zeros(4), torch.zeros(4), 1.0)


def test_range_rejects_bad_arguments_on_host(lib):
    f = lib.dit_attn_fwd_range
    assert f(A, B_, C, O, L, 1, 2, 256, 64, -1, 10, None) == INVALID
    assert f(A, B_, C, O, L, 1, 2, 256, 64, 0, 257, None) == INVALID          # j1 past S
    assert f(A, B_, C, O, L, 1, 2, 256, 64, 10, 10, None) == INVALID          # empty range
    assert f(A, B_, C, O, L, 1, 2, 256, 64, 20, 10, None) == INVALID
    assert f(A, B_, C, None, L, 1, 2, 256, 64, 0, 10, None) == INVALID
    assert f(A, B_, C, O, None, 1, 2, 256, 64, 0, 10, None) == INVALID
    assert f(A, B_, C, O + 4, L, 1, 2, 256, 64, 0, 10, None) == MISALIGNED
    assert f(A, B_, C, O, L, 1, 2, 256, 65, 0, 10, None) == SHAPE
    assert f(A, B_, C, B_ + 256, L, 1, 2, 256, 64, 0, 10, None) == INVALID    # out overlaps k
    assert f(A, B_, C, O, O + 64, 1, 2, 256, 64, 0, 10, None) == INVALID      # lse overlaps out


def test_torus_rejects_bad_arguments_on_host(lib):
    f = lib.dit_attn_fwd_torus
    KS, VS, K, V, P = 0x7F5000000000, 0x7F6000000000, 0x7F7000000000, 0x7F8000000000, 0x7F9000000000

    def call(q=A, ks=KS, vs=VS, k=K, v=V, p=P, ls=L, out=O, lo=None, S=256, D=64, n=4):
        return f(q, ks, vs, k, v, p, ls, out, lo, 1, 2, S, D, n, None, None)

    assert call(n=0) == INVALID
    assert call(n=65) == INVALID                  # more chunks than the event pool holds
    assert call(n=257) == INVALID                 # more chunks than keys
    assert call(ks=None) == INVALID
    assert call(vs=None) == INVALID
    assert call(p=None) == INVALID
    assert call(out=None) == INVALID
    assert call(D=96) == SHAPE
    assert call(p=P + 8) == MISALIGNED
    assert call(lo=L + 0x1000000 + 4) == MISALIGNED
    assert call(k=V) == INVALID                   # k and v the same buffer
    assert call(p=A) == INVALID                   # partials over q
    assert call(ks=K) == INVALID                  # source is the landing buffer
    assert call(ks=V) == INVALID                  # k_src is v: chunk copies into v overwrite it
    assert call(vs=K + 64) == INVALID             # v_src overlaps k
    assert call(ls=P + 64) == INVALID             # lses inside partials


def test_split_workspace_size_and_host_checks(lib):
    sz = lib.dit_attn_split_workspace_bytes
    rows, D, n = 2 * 16 * 1024, 72, 4
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert sz(2, 16, 1024, 72, 4) == up(n * rows * D * 4) + up(n * rows * 4)
    assert sz(2, 16, 1024, 65, 4) == 0 and sz(0, 16, 1024, 72, 4) == 0
    assert sz(2, 16, 1024, 72, 0) == 0 and sz(1, 1, 8, 64, 9) == 0   # n_split past S
    f = lib.dit_attn_fwd_split
    W = 0x7F5000000000
    nb = sz(1, 2, 256, 64, 2)

    def call(q=A, out=O, lse=L, ws=W, wsb=nb, S=256, D=64, ns=2):
        return f(q, B_, C, out, lse, 1, 2, S, D, ns, ws, wsb, None)

    assert call(ws=None) == INVALID
    assert call(out=None) == INVALID
    assert call(ns=0) == INVALID
    assert call(ns=257) == INVALID              # more chunks than keys
    assert call(wsb=nb - 1) == INVALID          # workspace too small
    assert call(ws=W + 8) == MISALIGNED
    assert call(lse=L + 2) == MISALIGNED
    assert call(ws=A + 64) == INVALID           # workspace over q
    assert call(ws=O) == INVALID                # workspace over out
    assert call(lse=W + 64) == INVALID          # lse inside the workspace
    assert call(D=96) == SHAPE


def test_split_rejects_partials_past_the_merge_limits(lib):
    # 2^47 partial elements: refused by the size query and the call alike
    assert lib.dit_attn_split_workspace_bytes(1, 1 << 14, 1 << 16, 128, 1 << 10) == 0
    assert lib.dit_attn_fwd_split(A, B_, C, O, L, 1, 1 << 14, 1 << 16, 128, 1 << 10,
                                  0x7F5000000000, 1 << 62, None) == INVALID
