"""Host loop of block-wise decoding over the C ABI's dllm_decode_step.

Per block (Sangam abstract: block-sized decodes with a recurring prefill;
dInfer article, "vicinity KV refresh"): reset the block state, one refresh
step (full forward, refills the K/V cache, first commit), then window steps
until every position of the block is committed. A window step recomputes
the window's K/V and attends over the whole sequence, the K/V outside the
window staying as the refresh left them (dual_cache, the default), or over
the cached prefix and the window only (dual_cache=False). Each step is one library
call that enqueues the whole step; the host reads back only the 4-byte
commit count to know when the block is done.
"""

from __future__ import annotations

import torch

from . import _binding as B


class BlockDecoder:
    """Device buffers and the step loop for one request.

    weights: dict with device bf16 tensors ``emb``, ``w_head`` ([V][d]) and
    per-layer lists ``wqkv`` ([3d][d]), ``wo``, ``wgu`` ([2 ffn][d]),
    ``wdown``, plus ``H``, ``rms_eps``, ``rope_base``.
    """

    def __init__(self, weights, prompt, *, resp_len, blk, vic, params, device="cuda", eos_id=-1,
                 dual_cache=True):
        dev = torch.device(device)
        self.weights = weights
        self.Lp = int(prompt.numel())
        self.T = self.Lp + int(resp_len)
        self.blk, self.vic = int(blk), int(vic)
        self.nblocks = int(resp_len) // self.blk
        self.params = dict(params)
        d = weights["emb"].shape[1]
        layers = len(weights["wqkv"])
        self.desc, self._keep = B.model_desc(weights, self.T)
        bf = torch.bfloat16
        self.k_cache = [torch.zeros((self.T, d), dtype=bf, device=dev) for _ in range(layers)]
        self.v_cache = [torch.zeros((self.T, d), dtype=bf, device=dev) for _ in range(layers)]
        self.tokens = torch.full((self.T,), int(params["mask_id"]), dtype=torch.int32, device=dev)
        self.tokens[:self.Lp] = prompt.to(dev, torch.int32)
        self.masked = torch.zeros(self.T, dtype=torch.uint8, device=dev)
        self.masked[self.Lp:] = 1
        b = self.blk
        self.bmask = torch.empty(b, dtype=torch.uint8, device=dev)
        self.btokens = torch.empty(b, dtype=torch.int32, device=dev)
        self.bprev = torch.empty(b, dtype=torch.int32, device=dev)
        self.bcredit = torch.empty(b, dtype=torch.float32, device=dev)
        self.bnext_emb = torch.zeros((b, d), dtype=bf, device=dev)
        self.n_commit = torch.zeros(1, dtype=torch.int32, device=dev)
        self.argmax = torch.empty(b, dtype=torch.int32, device=dev)
        self.conf = torch.empty(b, dtype=torch.float32, device=dev)
        self.pe = torch.empty((b, d), dtype=torch.float32, device=dev)
        self.hidden = torch.empty((b, d), dtype=bf, device=dev)
        self._kc = B._ptr_array(self.k_cache)
        self._vc = B._ptr_array(self.v_cache)
        P = B.ctypes.POINTER(B.c_void_p)
        self.state = B.DecodeState(
            self.T, self.Lp, self.blk, self.vic, self.tokens.data_ptr(), self.masked.data_ptr(),
            B.ctypes.cast(self._kc, P), B.ctypes.cast(self._vc, P), self.bmask.data_ptr(),
            self.btokens.data_ptr(), self.bprev.data_ptr(), self.bcredit.data_ptr(), self.bnext_emb.data_ptr(),
            self.n_commit.data_ptr(), self.argmax.data_ptr(), self.conf.data_ptr(), self.pe.data_ptr(),
            self.hidden.data_ptr(), B.params_struct(self.params), int(eos_id), int(bool(dual_cache)))
        self.eos_id = int(eos_id)
        self.ws = B.workspace(B.decode_step_workspace(self.desc, self.state), dev)
        self._graph = None

    def block_start(self, b):
        return self.Lp + b * self.blk

    def reset_block(self, b):
        b0 = self.block_start(b)
        self.bmask.copy_(self.masked[b0:b0 + self.blk])
        self.btokens.copy_(self.tokens[b0:b0 + self.blk])
        self.bprev.fill_(-1)
        self.bcredit.zero_()

    def step(self, b, refresh):
        B.decode_step(self.desc, self.state, b, refresh, self.ws)

    def restart(self, prompt=None):
        """Back to the initial sequence: the prompt, then a masked response."""
        if prompt is not None:
            self.tokens[:self.Lp].copy_(prompt, non_blocking=True)
        self.tokens[self.Lp:].fill_(int(self.params["mask_id"]))
        self.masked.zero_()
        self.masked[self.Lp:] = 1

    def eos_committed(self, upto):
        """Host check: a committed response position before `upto` holds eos_id."""
        if self.eos_id < 0 or upto <= self.Lp:
            return False
        seg = self.tokens[self.Lp:upto]
        live = self.masked[self.Lp:upto] == 0
        return bool(((seg == self.eos_id) & live).any().item())

    def decode_graph(self, stream=None):
        """The whole loop as one device-side CUDA graph (no host read per step)."""
        if self._graph is None:
            self._graph = B.DecodeGraph(self.desc, self.state, self.ws)
        self._graph.launch(stream)

    def decode(self, on_step=None, max_blocks=None):
        """Decode every block from the host; returns the number of steps per block."""
        steps_per_block = []
        for b in range(self.nblocks if max_blocks is None else min(max_blocks, self.nblocks)):
            if self.eos_committed(self.block_start(b)):
                break
            self.reset_block(b)
            remaining = int(self.bmask.sum().item())
            steps = 0
            while remaining > 0:
                if on_step is not None:
                    on_step("before", b, steps, self)
                self.step(b, refresh=(steps == 0))
                remaining -= int(self.n_commit.item())
                if on_step is not None:
                    on_step("after", b, steps, self)
                steps += 1
                if steps > self.blk:
                    raise RuntimeError("block did not finish in blk steps (at least one commit per step)")
            steps_per_block.append(steps)
        return steps_per_block
