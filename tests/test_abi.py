"""The C-ABI library: it loads, exports every function include/*.h declares,
and rejects bad arguments on the host before anything is launched (CPU only,
no GPU needed: validation runs before the first CUDA call)."""

import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT

import block_decoding_gb300 as bd


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"\b(dllm_[A-Za-z0-9_]+)\s*\(", src):
            names.add(m.group(1))
    return names


def test_exports_every_declared_symbol():
    names = _declared()
    assert {"dllm_block_attn", "dllm_head_confidence", "dllm_commit", "dllm_denoise_step"} <= names
    lib = ctypes.CDLL(bd.LIB_PATH)
    missing = [n for n in sorted(names) if not hasattr(lib, n)]
    assert not missing, missing
    # the binding declares a signature for every entry point
    assert names <= set(bd._binding.SIGNATURES)


def test_status_strings():
    assert bd.status_string(0) == "ok"
    for c in range(1, 6):
        assert bd.status_string(c) not in ("ok", "unknown status")
    assert bd.LIB.dllm_version() >= 1


P = ctypes.c_void_p


def test_commit_rejects_bad_arguments_on_host():
    L = bd.LIB
    prm = bd.Params(0.9, 0.7, 1.5, 1, 1, 1, 1.0, 5)
    fake = P(256)
    args = [fake] * 5 + [4, 1, 32] + [fake] * 5 + [16, 64] + [fake, fake]
    # NULL params
    assert L.dllm_commit(*args, None, None) == 1
    # blk > 64 unsupported
    a2 = list(args); a2[7] = 65
    assert L.dllm_commit(*a2, ctypes.byref(prm), None) == 2
    # mask_id outside [0, V)
    bad = bd.Params(0.9, 0.7, 1.5, 1, 1, 1, 1.0, 16)
    assert L.dllm_commit(*args, ctypes.byref(bad), None) == 1
    # hierarchical with zero levels
    bad = bd.Params(0.9, 0.7, 1.5, 1, 0, 1, 1.0, 5)
    assert L.dllm_commit(*args, ctypes.byref(bad), None) == 1
    # smoothing without P.E
    a3 = list(args); a3[2] = None
    assert L.dllm_commit(*a3, ctypes.byref(prm), None) == 1


def test_head_rejects_bad_arguments_on_host():
    L = bd.LIB
    fake = P(256)
    # d not a multiple of 64
    assert L.dllm_head_confidence(fake, fake, fake, 4, 100, 50, fake, fake, fake, fake, 1 << 30, None) == 2
    # P.E requested without an embedding table
    assert L.dllm_head_confidence(fake, fake, None, 4, 128, 50, fake, fake, fake, fake, 1 << 30, None) == 1
    # workspace too small
    assert L.dllm_head_confidence(fake, fake, fake, 4, 128, 50, fake, fake, fake, fake, 16, None) == 3
    # workspace misaligned
    need = L.dllm_head_workspace(4, 128, 50, 1)
    assert L.dllm_head_confidence(fake, fake, fake, 4, 128, 50, fake, fake, fake, P(256 + 16), need, None) == 3
    # nothing to do is fine and touches nothing
    assert L.dllm_head_confidence(None, None, None, 0, 128, 50, None, None, None, None, 0, None) == 0


def test_attention_rejects_bad_arguments_on_host():
    L = bd.LIB
    fake = P(256)
    ok = (1, 4, 64, 8, 8, 8, 8, 0.1, None, 0, None)
    assert L.dllm_block_attn(fake, fake, fake, fake, 0, fake, fake, 1, 4, 96, 8, 8, 8, 8, 0.1, None, 0, None) == 2
    assert L.dllm_block_attn(None, fake, fake, fake, 0, fake, fake, *ok) == 1
    assert L.dllm_block_attn(fake, fake, fake, fake, 0, fake, fake, -1, *ok[1:]) == 1
    assert L.dllm_block_attn(P(258), fake, fake, fake, 0, fake, fake, *ok) == 1
    assert L.dllm_block_attn(fake, fake, fake, fake, 0, fake, fake, 1, 4, 64, 8, 8, -1, 8, 0.1, None, 0, None) == 1


def test_denoise_step_checks_workspace_on_host():
    a = bd.StepArgs()
    a.R, a.d, a.V, a.B, a.blk = 4, 128, 100, 1, 4
    need = bd.denoise_step_workspace(a)
    assert need >= 4 * 100 * 4
    rc = bd.LIB.dllm_denoise_step(ctypes.byref(a), None, 0, None)
    assert rc == 3


@pytest.mark.parametrize("R,d,V", [(1, 64, 1), (32, 4096, 126464), (512, 4096, 126464)])
def test_workspace_sizes_are_aligned_and_monotone(R, d, V):
    w0 = bd.head_workspace(R, d, V, 0)
    w1 = bd.head_workspace(R, d, V, 1)
    assert w0 % 256 == 0 and w1 % 256 == 0 and w1 >= w0 > 0


def test_moe_rejects_bad_arguments_on_host():
    L = bd.LIB
    fake = P(256)
    w = [fake] * 4

    def call(n=8, d=256, E=8, F=128, k=2, ptrs=w, out=fake, ws=fake, ws_bytes=1 << 30):
        return L.dllm_moe_ffn(*ptrs, n, d, E, F, k, out, 1, None, None, ws, ws_bytes, None)

    assert call(d=100) == 2                 # d not a multiple of 128
    assert call(F=64) == 2                  # F not a multiple of 128
    assert call(E=0) == 2 and call(E=300) == 2
    assert call(k=9) == 2 and call(k=17, E=32) == 2   # topk > E, topk > 16
    assert call(n=40000, k=2) == 2          # more than 65536 assignments
    assert call(ptrs=[None] + w[1:]) == 1   # null input
    assert call(ptrs=[P(258)] + w[1:]) == 1  # misaligned input
    assert call(ws_bytes=16) == 3           # workspace too small
    assert call(ws=P(256 + 16)) == 3        # workspace misaligned
    assert call(n=0, ptrs=[None] * 4, out=None, ws=None, ws_bytes=0) == 0   # nothing to do
    assert L.dllm_moe_ffn_workspace(8, 256, 8, 128, 2) % 256 == 0
    assert L.dllm_moe_ffn_workspace(8, 100, 8, 128, 2) == 0


def test_attention_workspace_bound_is_monotone_and_small():
    W = bd.LIB.dllm_block_attn_workspace
    assert W(1, 4, 64, 32, 128) == 0                      # one key tile: never split
    for dh in (64, 128):
        prev = 0
        for kv in (256, 512, 1024, 8384):
            cur = W(1, 32, dh, 96, kv)
            assert cur >= prev and cur % 256 == 0
            prev = cur
            # any smaller query bound fits in the larger one's workspace
            assert all(W(1, 32, dh, q, kv) <= W(1, 32, dh, 512, kv) for q in (1, 96, 200, 512))
        assert W(16, 32, dh, 8384, 8384) <= 256 * 128 * (dh * 4 + 8) + 512   # 256 CTAs x 128 query rows


def test_workspace_bytes_matches_the_per_call_sizes():
    W = bd.LIB.dllm_workspace_bytes
    assert W(0, 2, 32, 128, 96, 608, 0, 0, 0) == bd.LIB.dllm_block_attn_workspace(2, 32, 128, 96, 608)
    assert W(1, 0, 0, 0, 0, 0, 32, 4096, 126464) == bd.head_workspace(32, 4096, 126464, 0)
    assert W(2, 0, 0, 0, 0, 0, 32, 4096, 126464) == bd.head_workspace(32, 4096, 126464, 1)
    a = bd.StepArgs()
    a.attn_out, a.pe = 1, 1
    a.B, a.H, a.dh, a.max_q, a.max_kv, a.R, a.d, a.V = 1, 32, 128, 96, 608, 32, 4096, 126464
    assert W(3, 1, 32, 128, 96, 608, 32, 4096, 126464) == bd.denoise_step_workspace(a)
    assert W(9, 1, 1, 64, 1, 1, 1, 64, 2) == 0
