"""Upload a workload to the GPU and run the library on it (test infrastructure)."""

import numpy as np
import torch

import block_decoding_gb300 as bd
from helpers import dev, dev_bf16, host_bf16_bits


def upload_step(inp, attn_fp32=True):
    g = dict(
        q=dev_bf16(inp["q"]), k=dev_bf16(inp["k"]), v=dev_bf16(inp["v"]),
        q_off=dev(inp["q_off"]), kv_off=dev(inp["kv_off"]),
        w_head=dev_bf16(inp["w_head"]), emb=dev_bf16(inp["emb"]),
        hidden=dev_bf16(inp["hidden"]),
        row_req=dev(inp["row_req"]), row_pos=dev(inp["row_pos"]),
        mask=dev(inp["mask"]), tokens=dev(inp["tokens"]),
        credit=dev(inp["credit"]), prev=dev(inp["prev"]),
    )
    R, d, B, blk = inp["R"], inp["d"], inp["B"], inp["blk"]
    g["attn_out"] = torch.empty(g["q"].shape, dtype=torch.float32 if attn_fp32 else torch.bfloat16,
                                device="cuda")
    g["argmax"] = torch.empty(R, dtype=torch.int32, device="cuda")
    g["conf"] = torch.empty(R, dtype=torch.float32, device="cuda")
    g["pe"] = torch.empty((R, d), dtype=torch.float32, device="cuda") if inp["params"]["smoothing"] else None
    g["next_emb"] = torch.empty((B, blk, d), dtype=torch.bfloat16, device="cuda")
    g["n_commit"] = torch.empty(B, dtype=torch.int32, device="cuda")
    return g


def step_args(inp, g, with_attention=True):
    kw = {}
    if with_attention:
        kw = dict(q=g["q"], k=g["k"], v=g["v"], attn_out=g["attn_out"], q_off=g["q_off"],
                  kv_off=g["kv_off"], max_q=inp["max_q"], max_kv=inp["max_kv"], scale=inp["scale"])
    return bd.step_args(hidden=g["hidden"], w_head=g["w_head"], emb=g["emb"], argmax=g["argmax"],
                        conf=g["conf"], pe=g["pe"], row_req=g["row_req"], row_pos=g["row_pos"],
                        mask=g["mask"], tokens=g["tokens"], credit=g["credit"], prev=g["prev"],
                        next_emb=g["next_emb"], n_commit=g["n_commit"], params=inp["params"], **kw)


def run_step(inp, g=None, with_attention=True):
    """One dllm_denoise_step; returns host copies of every output."""
    g = g or upload_step(inp)
    a = step_args(inp, g, with_attention)
    ws = bd.workspace(bd.denoise_step_workspace(a))
    bd.denoise_step(a, ws)
    torch.cuda.synchronize()
    st = bd.device_status()
    assert st == 0, f"device status {st:#x}"
    return host_state(g, with_attention)


def host_state(g, with_attention=True):
    out = dict(
        argmax=g["argmax"].cpu().numpy(), conf=g["conf"].cpu().numpy(),
        pe=g["pe"].cpu().numpy() if g["pe"] is not None else None,
        mask=g["mask"].cpu().numpy(), tokens=g["tokens"].cpu().numpy(),
        credit=g["credit"].cpu().numpy(), prev=g["prev"].cpu().numpy(),
        n_commit=g["n_commit"].cpu().numpy(), next_emb_bits=host_bf16_bits(g["next_emb"]),
    )
    if with_attention:
        o = g["attn_out"]
        out["attn"] = (o.cpu().numpy() if o.dtype == torch.float32
                       else o.float().cpu().numpy())
    return out
