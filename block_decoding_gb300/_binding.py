"""ctypes binding of libdllm.so: argument marshalling only.

Every function takes torch CUDA tensors (PyTorch supplies device memory and
streams), checks dtype / contiguity / device, and passes raw pointers and
sizes to the C ABI declared in ``include/dllm.h``. All arithmetic of the
denoise step runs in the library's kernels; there is no fallback path: a
missing library raises at import time.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdllm.so")

c_int, c_float, c_size_t, c_void_p = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p


class DllmError(RuntimeError):
    def __init__(self, code, what):
        msg = f"{what}: {status_string(code)} (status {code})"
        if code == 4:
            name = LIB.dllm_last_cuda_error()
            if name:
                msg += f": {name.decode()}"
        super().__init__(msg)
        self.code = code


class Params(ctypes.Structure):
    _fields_ = [("tau", c_float), ("lambda_", c_float), ("kappa", c_float),
                ("hierarchical", c_int), ("hier_levels", c_int), ("smoothing", c_int),
                ("alpha", c_float), ("mask_id", c_int)]


class StepArgs(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("k", c_void_p), ("v", c_void_p),
                ("attn_out", c_void_p), ("attn_out_fp32", c_int),
                ("q_off", c_void_p), ("kv_off", c_void_p),
                ("H", c_int), ("dh", c_int), ("max_q", c_int), ("max_kv", c_int),
                ("q_rows", c_int), ("kv_rows", c_int),
                ("scale", c_float),
                ("hidden", c_void_p), ("w_head", c_void_p), ("emb", c_void_p),
                ("R", c_int), ("d", c_int), ("V", c_int),
                ("argmax", c_void_p), ("conf", c_void_p), ("pe", c_void_p),
                ("row_req", c_void_p), ("row_pos", c_void_p),
                ("B", c_int), ("blk", c_int),
                ("mask", c_void_p), ("tokens", c_void_p), ("credit", c_void_p),
                ("prev_argmax", c_void_p), ("next_emb", c_void_p), ("n_commit", c_void_p),
                ("params", Params)]


# name -> (restype, argtypes); mirrors include/dllm.h
SIGNATURES = {
    "dllm_block_attn_workspace": (c_size_t, [c_int] * 5),
    "dllm_block_attn": (c_int, [c_void_p] * 4 + [c_int, c_void_p, c_void_p] + [c_int] * 7
                        + [c_float, c_void_p, c_size_t, c_void_p]),
    "dllm_head_workspace": (c_size_t, [c_int] * 4),
    "dllm_head_confidence": (c_int, [c_void_p] * 3 + [c_int] * 3 + [c_void_p] * 4
                             + [c_size_t, c_void_p]),
    "dllm_head_confidence_noalloc": (c_int, [c_void_p] * 3 + [c_int] * 3 + [c_void_p] * 4),
    "dllm_commit": (c_int, [c_void_p] * 5 + [c_int] * 3 + [c_void_p] * 5 + [c_int, c_int]
                    + [c_void_p, c_void_p, ctypes.POINTER(Params), c_void_p]),
    "dllm_denoise_step_workspace": (c_size_t, [ctypes.POINTER(StepArgs)]),
    "dllm_workspace_bytes": (c_size_t, [c_int] * 9),
    "dllm_denoise_step": (c_int, [ctypes.POINTER(StepArgs), c_void_p, c_size_t, c_void_p]),
    "dllm_status_string": (ctypes.c_char_p, [c_int]),
    "dllm_get_device_status": (c_int, [ctypes.POINTER(ctypes.c_int32), c_int]),
    "dllm_last_cuda_error": (ctypes.c_char_p, []),
    "dllm_version": (c_int, []),
    "dllm_launch_count": (ctypes.c_uint64, []),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with block_decoding_gb300.build.build() "
            "(nvcc, sm_103a). There is no fallback implementation.")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


LIB = _load()


def launch_count() -> int:
    """Kernels this library has enqueued since it was loaded."""
    return int(LIB.dllm_launch_count())


def status_string(code: int) -> str:
    return LIB.dllm_status_string(int(code)).decode()


def _ck(code, what):
    if code != 0:
        raise DllmError(code, what)


def device_status(clear: bool = True) -> int:
    out = ctypes.c_int32(0)
    LIB.dllm_get_device_status(ctypes.byref(out), 1 if clear else 0)
    return int(out.value)


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not (isinstance(t, torch.Tensor) and t.is_cuda):
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def params_struct(p: dict) -> Params:
    return Params(float(p["tau"]), float(p["lam"]), float(p["kappa"]),
                  int(p["hierarchical"]), int(p["hier_levels"]), int(p["smoothing"]),
                  float(p["alpha"]), int(p["mask_id"]))


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A caller-owned workspace buffer (torch allocations are 256-byte aligned)."""
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device or "cuda")


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------

def block_attn_workspace(B, H, dh, max_q, max_kv) -> int:
    return int(LIB.dllm_block_attn_workspace(B, H, dh, max_q, max_kv))


def block_attn(q, k, v, q_off, kv_off, max_q, max_kv, scale=None, out=None,
               out_fp32=False, ws=None, stream=None):
    """Non-causal block attention; q [sum W][H][dh], k/v [sum L][H][dh] bf16."""
    H, dh = q.shape[1], q.shape[2]
    B = q_off.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(dh)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32 if out_fp32 else torch.bfloat16, device=q.device)
    need = block_attn_workspace(B, H, dh, max_q, max_kv)
    if ws is None and need:
        ws = workspace(need, q.device)
    rc = LIB.dllm_block_attn(_ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"),
                             _ptr(v, torch.bfloat16, "v"), _ptr(out, None, "out"),
                             1 if out.dtype == torch.float32 else 0,
                             _ptr(q_off, torch.int32, "q_off"), _ptr(kv_off, torch.int32, "kv_off"),
                             B, H, dh, int(max_q), int(max_kv), q.shape[0], k.shape[0], float(scale),
                             _ptr(ws, None, "ws") if ws is not None else None,
                             ws.numel() if ws is not None else 0, _stream(stream))
    _ck(rc, "dllm_block_attn")
    return out


def head_workspace(R, d, V, with_pe) -> int:
    return int(LIB.dllm_head_workspace(R, d, V, 1 if with_pe else 0))


def head_confidence(hidden, w_head, emb=None, with_pe=True, argmax=None, conf=None,
                    pe=None, ws=None, stream=None):
    """LM head + softmax stats (+ P.E); returns (argmax int32, conf f32, pe f32 or None)."""
    R, d = hidden.shape
    V = w_head.shape[0]
    dev = hidden.device
    with_pe = with_pe and emb is not None
    argmax = argmax if argmax is not None else torch.empty(R, dtype=torch.int32, device=dev)
    conf = conf if conf is not None else torch.empty(R, dtype=torch.float32, device=dev)
    if with_pe and pe is None:
        pe = torch.empty((R, d), dtype=torch.float32, device=dev)
    if not with_pe:
        pe = None
    need = head_workspace(R, d, V, with_pe)
    if ws is None:
        ws = workspace(need, dev)
    rc = LIB.dllm_head_confidence(_ptr(hidden, torch.bfloat16, "hidden"),
                                  _ptr(w_head, torch.bfloat16, "w_head"),
                                  _ptr(emb, torch.bfloat16, "emb") if emb is not None else None,
                                  R, d, V, _ptr(argmax, torch.int32, "argmax"),
                                  _ptr(conf, torch.float32, "conf"),
                                  _ptr(pe, torch.float32, "pe") if pe is not None else None,
                                  _ptr(ws, None, "ws"), ws.numel(), _stream(stream))
    _ck(rc, "dllm_head_confidence")
    return argmax, conf, pe


def commit(argmax, conf, pe, row_req, row_pos, mask, tokens, credit, prev, emb,
           params: dict, next_emb=None, n_commit=None, stream=None):
    """Parallel-decode commit; updates mask/tokens/credit/prev in place."""
    B, blk = mask.shape
    V, d = emb.shape
    R = row_req.numel()
    dev = mask.device
    next_emb = next_emb if next_emb is not None else torch.empty((B, blk, d), dtype=torch.bfloat16, device=dev)
    n_commit = n_commit if n_commit is not None else torch.empty(B, dtype=torch.int32, device=dev)
    prm = params_struct(params)
    rc = LIB.dllm_commit(_ptr(argmax, torch.int32, "argmax"), _ptr(conf, torch.float32, "conf"),
                         _ptr(pe, torch.float32, "pe") if pe is not None else None,
                         _ptr(row_req, torch.int32, "row_req"), _ptr(row_pos, torch.int32, "row_pos"),
                         R, B, blk, _ptr(mask, torch.uint8, "mask"), _ptr(tokens, torch.int32, "tokens"),
                         _ptr(credit, torch.float32, "credit"), _ptr(prev, torch.int32, "prev"),
                         _ptr(emb, torch.bfloat16, "emb"), V, d,
                         _ptr(next_emb, torch.bfloat16, "next_emb"), _ptr(n_commit, torch.int32, "n_commit"),
                         ctypes.byref(prm), _stream(stream))
    _ck(rc, "dllm_commit")
    return next_emb, n_commit


def step_args(*, q=None, k=None, v=None, attn_out=None, q_off=None, kv_off=None,
              max_q=0, max_kv=0, scale=None, hidden, w_head, emb, argmax, conf, pe,
              row_req, row_pos, mask, tokens, credit, prev, next_emb, n_commit,
              params: dict) -> StepArgs:
    a = StepArgs()
    if attn_out is not None:
        a.q, a.k, a.v = _ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"), _ptr(v, torch.bfloat16, "v")
        a.attn_out = _ptr(attn_out, None, "attn_out")
        a.attn_out_fp32 = 1 if attn_out.dtype == torch.float32 else 0
        a.q_off, a.kv_off = _ptr(q_off, torch.int32, "q_off"), _ptr(kv_off, torch.int32, "kv_off")
        a.H, a.dh = q.shape[1], q.shape[2]
        a.max_q, a.max_kv = int(max_q), int(max_kv)
        a.q_rows, a.kv_rows = q.shape[0], k.shape[0]
        a.scale = float(scale if scale is not None else 1.0 / math.sqrt(a.dh))
    a.hidden = _ptr(hidden, torch.bfloat16, "hidden")
    a.w_head = _ptr(w_head, torch.bfloat16, "w_head")
    a.emb = _ptr(emb, torch.bfloat16, "emb")
    a.R, a.d = hidden.shape
    a.V = w_head.shape[0]
    a.argmax, a.conf = _ptr(argmax, torch.int32, "argmax"), _ptr(conf, torch.float32, "conf")
    a.pe = _ptr(pe, torch.float32, "pe") if pe is not None else None
    a.row_req, a.row_pos = _ptr(row_req, torch.int32, "row_req"), _ptr(row_pos, torch.int32, "row_pos")
    a.B, a.blk = mask.shape
    a.mask = _ptr(mask, torch.uint8, "mask")
    a.tokens = _ptr(tokens, torch.int32, "tokens")
    a.credit = _ptr(credit, torch.float32, "credit")
    a.prev_argmax = _ptr(prev, torch.int32, "prev")
    a.next_emb = _ptr(next_emb, torch.bfloat16, "next_emb")
    a.n_commit = _ptr(n_commit, torch.int32, "n_commit")
    a.params = params_struct(params)
    return a


def denoise_step_workspace(args: StepArgs) -> int:
    return int(LIB.dllm_denoise_step_workspace(ctypes.byref(args)))


def denoise_step(args: StepArgs, ws, stream=None):
    rc = LIB.dllm_denoise_step(ctypes.byref(args), _ptr(ws, None, "ws"), ws.numel(), _stream(stream))
    _ck(rc, "dllm_denoise_step")


# ---------------------------------------------------------------------------
# end-to-end model (dllm_gemm_bf16, dllm_model_forward, dllm_decode_step)
# ---------------------------------------------------------------------------

class ModelDesc(ctypes.Structure):
    _fields_ = [("layers", c_int), ("d", c_int), ("H", c_int), ("dh", c_int), ("ffn", c_int), ("V", c_int),
                ("max_seq", c_int), ("rms_eps", c_float), ("rope_base", c_float),
                ("emb", c_void_p), ("w_head", c_void_p),
                ("wqkv", ctypes.POINTER(c_void_p)), ("wo", ctypes.POINTER(c_void_p)),
                ("wgu", ctypes.POINTER(c_void_p)), ("wdown", ctypes.POINTER(c_void_p))]


class DecodeState(ctypes.Structure):
    _fields_ = [("T", c_int), ("prompt_len", c_int), ("blk", c_int), ("vic", c_int),
                ("tokens", c_void_p), ("masked", c_void_p),
                ("k_cache", ctypes.POINTER(c_void_p)), ("v_cache", ctypes.POINTER(c_void_p)),
                ("bmask", c_void_p), ("btokens", c_void_p), ("bprev", c_void_p), ("bcredit", c_void_p),
                ("bnext_emb", c_void_p), ("n_commit", c_void_p), ("argmax", c_void_p), ("conf", c_void_p),
                ("pe", c_void_p), ("hidden", c_void_p), ("params", Params), ("eos_id", c_int),
                ("dual_cache", c_int)]


SIGNATURES.update({
    "dllm_gemm_bf16": (c_int, [c_void_p] * 3 + [c_int] * 4 + [c_void_p, c_void_p]),
    "dllm_model_forward_workspace": (c_size_t, [ctypes.POINTER(ModelDesc), c_int]),
    "dllm_model_forward": (c_int, [ctypes.POINTER(ModelDesc), c_void_p, c_int, c_int,
                                   ctypes.POINTER(c_void_p), ctypes.POINTER(c_void_p), c_void_p, c_void_p,
                                   c_size_t, c_void_p]),
    "dllm_decode_step_workspace": (c_size_t, [ctypes.POINTER(ModelDesc), ctypes.POINTER(DecodeState)]),
    "dllm_decode_step": (c_int, [ctypes.POINTER(ModelDesc), ctypes.POINTER(DecodeState), c_int, c_int,
                                 c_void_p, c_size_t, c_void_p]),
    "dllm_decode_graph_create": (c_int, [ctypes.POINTER(ModelDesc), ctypes.POINTER(DecodeState), c_void_p,
                                         c_size_t, ctypes.POINTER(c_void_p)]),
    "dllm_decode_graph_launch": (c_int, [c_void_p, c_void_p]),
    "dllm_decode_graph_destroy": (c_int, [c_void_p]),
})
for _name in ("dllm_gemm_bf16", "dllm_model_forward_workspace", "dllm_model_forward",
              "dllm_decode_step_workspace", "dllm_decode_step", "dllm_decode_graph_create",
              "dllm_decode_graph_launch", "dllm_decode_graph_destroy"):
    _fn = getattr(LIB, _name)
    _fn.restype, _fn.argtypes = SIGNATURES[_name]


def gemm_bf16(A, W, epilogue=0, aux=None, out=None, stream=None):
    """C = A W^T (+aux) or SwiGLU; A [M][K], W [N][K] (or [2N][K] for SwiGLU)."""
    M, K = A.shape
    N = W.shape[0] // 2 if epilogue == 2 else W.shape[0]
    out = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    rc = LIB.dllm_gemm_bf16(_ptr(A, torch.bfloat16, "A"), _ptr(W, torch.bfloat16, "W"),
                            _ptr(out, torch.bfloat16, "C"), M, N, K, int(epilogue),
                            _ptr(aux, torch.bfloat16, "aux") if aux is not None else None, _stream(stream))
    _ck(rc, "dllm_gemm_bf16")
    return out


def _ptr_array(tensors):
    arr = (c_void_p * len(tensors))(*[_ptr(t, torch.bfloat16, "weight") for t in tensors])
    return arr


def model_desc(weights: dict, max_seq: int):
    """ModelDesc over device weights: emb, w_head and per-layer lists wqkv/wo/wgu/wdown.

    Returns (desc, keepalive) -- keep the second value alive while desc is used.
    """
    L = len(weights["wqkv"])
    arrs = [_ptr_array(weights[k]) for k in ("wqkv", "wo", "wgu", "wdown")]
    d = weights["emb"].shape[1]
    desc = ModelDesc(L, d, weights["H"], d // weights["H"], weights["wgu"][0].shape[0] // 2,
                     weights["emb"].shape[0], int(max_seq), float(weights["rms_eps"]),
                     float(weights["rope_base"]), _ptr(weights["emb"], torch.bfloat16, "emb"),
                     _ptr(weights["w_head"], torch.bfloat16, "w_head"),
                     ctypes.cast(arrs[0], ctypes.POINTER(c_void_p)), ctypes.cast(arrs[1], ctypes.POINTER(c_void_p)),
                     ctypes.cast(arrs[2], ctypes.POINTER(c_void_p)), ctypes.cast(arrs[3], ctypes.POINTER(c_void_p)))
    return desc, arrs


def model_forward(desc, x_in, pos0, k_cache, v_cache, ws=None, stream=None):
    n = x_in.shape[0]
    need = int(LIB.dllm_model_forward_workspace(ctypes.byref(desc), n))
    ws = ws if ws is not None else workspace(need, x_in.device)
    out = torch.empty_like(x_in)
    kc, vc = _ptr_array(k_cache), _ptr_array(v_cache)
    rc = LIB.dllm_model_forward(ctypes.byref(desc), _ptr(x_in, torch.bfloat16, "x_in"), n, int(pos0),
                                ctypes.cast(kc, ctypes.POINTER(c_void_p)), ctypes.cast(vc, ctypes.POINTER(c_void_p)),
                                _ptr(out, torch.bfloat16, "hidden_out"), _ptr(ws, None, "ws"), ws.numel(),
                                _stream(stream))
    _ck(rc, "dllm_model_forward")
    return out


def decode_step_workspace(desc, state) -> int:
    return int(LIB.dllm_decode_step_workspace(ctypes.byref(desc), ctypes.byref(state)))


def decode_step(desc, state, block, refresh, ws, stream=None):
    rc = LIB.dllm_decode_step(ctypes.byref(desc), ctypes.byref(state), int(block), 1 if refresh else 0,
                              _ptr(ws, None, "ws"), ws.numel(), _stream(stream))
    _ck(rc, "dllm_decode_step")


class DecodeGraph:
    """One CUDA graph that runs the whole block decode loop on the device."""

    def __init__(self, desc, state, ws):
        h = c_void_p()
        rc = LIB.dllm_decode_graph_create(ctypes.byref(desc), ctypes.byref(state), _ptr(ws, None, "ws"),
                                          ws.numel(), ctypes.byref(h))
        _ck(rc, "dllm_decode_graph_create")
        self.handle = h

    def launch(self, stream=None):
        _ck(LIB.dllm_decode_graph_launch(self.handle, _stream(stream)), "dllm_decode_graph_launch")

    def close(self):
        if self.handle:
            LIB.dllm_decode_graph_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---------------------------------------------------------------------------
# step-level scheduler (include/dllm_sched.h): host-only
# ---------------------------------------------------------------------------
class SchedConfig(ctypes.Structure):
    _fields_ = [("slots", c_int), ("blk", c_int), ("vic", c_int), ("quantum", c_int), ("budget_cap", c_int),
                ("max_step_rows", c_int), ("max_seq", c_int), ("policy", c_int), ("dual_cache", c_int)]


class SchedEntry(ctypes.Structure):
    _fields_ = [("slot", c_int), ("req", c_int), ("block", c_int), ("kind", c_int), ("q_pos0", c_int),
                ("q_rows", c_int), ("kv_rows", c_int), ("b0", c_int)]


_I32P = ctypes.POINTER(ctypes.c_int32)
SIGNATURES.update({
    "dllm_sched_create": (c_int, [ctypes.POINTER(SchedConfig), ctypes.POINTER(c_void_p)]),
    "dllm_sched_destroy": (None, [c_void_p]),
    "dllm_sched_submit": (c_int, [c_void_p, c_int, c_int, c_int]),
    "dllm_sched_plan": (c_int, [c_void_p, ctypes.POINTER(SchedEntry), c_int]),
    "dllm_sched_complete": (c_int, [c_void_p, _I32P, ctypes.POINTER(ctypes.c_uint8)]),
    "dllm_sched_budget": (ctypes.c_longlong, [c_void_p]),
    "dllm_sched_queued": (c_int, [c_void_p]),
    "dllm_sched_finished": (c_int, [c_void_p, _I32P, c_int]),
    "dllm_sched_pack": (c_int, [ctypes.POINTER(SchedEntry), c_int, c_int, c_int, _I32P, _I32P, _I32P, _I32P]),
})
for _name in ("dllm_sched_create", "dllm_sched_destroy", "dllm_sched_submit", "dllm_sched_plan",
              "dllm_sched_complete", "dllm_sched_budget", "dllm_sched_queued", "dllm_sched_finished",
              "dllm_sched_pack"):
    _fn = getattr(LIB, _name)
    _fn.restype, _fn.argtypes = SIGNATURES[_name]


# ---------------------------------------------------------------------------
# mixture-of-experts FFN (dllm_moe_ffn)
# ---------------------------------------------------------------------------
SIGNATURES.update({
    "dllm_moe_ffn_workspace": (c_size_t, [c_int] * 5),
    "dllm_moe_ffn": (c_int, [c_void_p] * 4 + [c_int] * 5 + [c_void_p, c_int, c_void_p, c_void_p, c_void_p,
                                                           c_size_t, c_void_p]),
})
for _name in ("dllm_moe_ffn_workspace", "dllm_moe_ffn"):
    _fn = getattr(LIB, _name)
    _fn.restype, _fn.argtypes = SIGNATURES[_name]


def moe_ffn(h, w_router, w13, w2, topk, out_fp32=True, out=None, ids=None, weights=None, ws=None, stream=None):
    """out [n][d] = top-k MoE SwiGLU FFN of h; returns (out, ids, weights).
    w13 [E][2F][d] (gate rows, then up rows per expert), w2 [E][d][F]."""
    n, d = h.shape
    E, F2, d2 = w13.shape
    F = F2 // 2
    if d2 != d or tuple(w2.shape) != (E, d, F) or tuple(w_router.shape) != (E, d):
        raise ValueError("moe_ffn: inconsistent shapes")
    dev = h.device
    if out is None:
        out = torch.empty((n, d), dtype=torch.float32 if out_fp32 else torch.bfloat16, device=dev)
    if ids is None:
        ids = torch.empty((n, topk), dtype=torch.int32, device=dev)
    if weights is None:
        weights = torch.empty((n, topk), dtype=torch.float32, device=dev)
    need = int(LIB.dllm_moe_ffn_workspace(n, d, E, F, topk))
    if need == 0 and n > 0:
        raise DllmError(2, "dllm_moe_ffn_workspace")
    if ws is None or ws.numel() < need:
        ws = workspace(max(need, 256), dev)
    rc = LIB.dllm_moe_ffn(_ptr(h, torch.bfloat16, "h"), _ptr(w_router, torch.bfloat16, "w_router"),
                          _ptr(w13, torch.bfloat16, "w13"), _ptr(w2, torch.bfloat16, "w2"), n, d, E, F, topk,
                          _ptr(out, None, "out"), 1 if out.dtype == torch.float32 else 0,
                          _ptr(ids, torch.int32, "ids"), _ptr(weights, torch.float32, "weights"),
                          _ptr(ws, None, "ws"), ws.numel(), _stream(stream))
    _ck(rc, "dllm_moe_ffn")
    return out, ids, weights
