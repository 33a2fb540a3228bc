"""The allocation-free head entry point (GPU).

dllm_head_confidence_noalloc serves callers that cannot call cudaMalloc or
keep a workspace of their own (for example a plugin whose host framework
owns all device memory, or a thread that must not block on an allocation):
its scratch is a fixed device array inside the library. This file checks it
through the C ABI against dllm_head_confidence with a caller workspace, on
two calls in a row with different inputs (the array keeps the previous
call's contents, which must not leak into the next result), and that an
oversized request is refused before anything runs. Both calls are also
checked against the oracle's head (argmax exact outside near-ties,
confidence and P.E within the parity tolerances), so a scratch-layout fault
that both entry points shared would still be caught. It is named to be
collected last, and passes alone in a fresh process too: the first call on
the device performs the array's one-time address look-up.
"""

import ctypes

import numpy as np
import pytest
import torch

import block_decoding_gb300 as bd
import oracle
from helpers import dev_bf16, rownorm_rel
from parity import CONF_TOL, PE_TOL, check_head
from workloads import bf16_bits_to_f64, make_step_inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _noalloc(hidden, w_head, emb, R, d, V):
    argmax = torch.empty(R, dtype=torch.int32, device="cuda")
    conf = torch.empty(R, dtype=torch.float32, device="cuda")
    pe = torch.empty((R, d), dtype=torch.float32, device="cuda")
    rc = bd.LIB.dllm_head_confidence_noalloc(hidden.data_ptr(), w_head.data_ptr(), emb.data_ptr(), R, d, V,
                                             argmax.data_ptr(), conf.data_ptr(), pe.data_ptr(),
                                             torch.cuda.current_stream().cuda_stream)
    assert rc == 0, bd.status_string(rc)
    return argmax, conf, pe


@pytest.mark.parametrize("H,V", [(4, 2048), (16, 32768)])
def test_noalloc_matches_workspace_entry_point_twice(H, V):
    inp = make_step_inputs(B=2, H=H, dh=64, V=V, blk=16, P=0, seed=21, cal=True)
    R, d = inp["R"], inp["d"]
    w_head, emb = dev_bf16(inp["w_head"]), dev_bf16(inp["emb"])
    rng = np.random.default_rng(0)
    second = inp["hidden"][rng.permutation(R)]           # a different input for call 2
    w64, e64 = bf16_bits_to_f64(inp["w_head"]), bf16_bits_to_f64(inp["emb"])
    for hid_bits in (inp["hidden"], second):
        hidden = dev_bf16(hid_bits)
        a_ref, c_ref, pe_ref = bd.head_confidence(hidden, w_head, emb)
        a, c, pe = _noalloc(hidden, w_head, emb, R, d, V)
        torch.cuda.synchronize()
        assert bd.device_status() == 0
        assert np.array_equal(a.cpu().numpy(), a_ref.cpu().numpy())
        assert np.abs(c.cpu().numpy() - c_ref.cpu().numpy()).max() <= CONF_TOL
        assert rownorm_rel(pe.cpu().numpy(), pe_ref.cpu().numpy()).max() <= PE_TOL
        ref = oracle.head_confidence(bf16_bits_to_f64(hid_bits), w64, e64)
        gap, sc = oracle.step.top2_gap(ref["z"])
        check_head(a.cpu().numpy(), c.cpu().numpy(), pe.cpu().numpy(), ref,
                   amb_rows=gap < oracle.step.ARGMAX_GAP_REL * sc)


def test_noalloc_rejects_oversized_requests():
    limit = int(ctypes.c_uint32(48 << 20).value)
    R, d, V = 512, 4096, 126464
    assert bd.head_workspace(R, d, V, True) > limit
    fake = 256
    rc = bd.LIB.dllm_head_confidence_noalloc(fake, fake, fake, R, d, V, fake, fake, fake, None)
    assert rc == 2      # DLLM_ERR_UNSUPPORTED, nothing launched
    assert bd.head_workspace(32, 4096, 126464, True) <= limit
