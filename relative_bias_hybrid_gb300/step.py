"""One pass of the hot path for a workload: prologue, then prefill or decode + combine.

Plumbing only: this module allocates the output buffers with torch, fills the params
structs through the binding and issues the C-ABI calls in order on one stream.
"""
from __future__ import annotations

from typing import Dict, Optional

import torch

from . import inkattn as ia
from .inputs import Workload


class AttentionStep:
    """Buffers + calls of one attention-layer pass over device-resident inputs.

    mode "prefill": inkattn_prologue then inkattn_prefill (inkattn_prefill_e4m3 over an
                    E4M3 cache, with its workspace).
    mode "decode":  inkattn_prologue then inkattn_decode (+ inkattn_combine when the
                    split count is above one).
    The conv state and the KV cache in `inputs` are updated in place by every run.
    """

    def __init__(self, w: Workload, inputs: Dict[str, torch.Tensor], mode: str = "prefill",
                 num_splits: int = 0, with_lse: bool = True, out_dtype=torch.bfloat16):
        if mode not in ("prefill", "decode"):
            raise ValueError(mode)
        self.w, self.x, self.mode = w, inputs, mode
        dev = inputs["q"].device
        N, Hq, d = inputs["q"].shape
        self.q_out = torch.empty_like(inputs["q"])
        self.out = torch.empty((N, Hq, d), dtype=out_dtype, device=dev)
        self.lse = torch.empty((N, Hq), dtype=torch.float32, device=dev) if with_lse else None
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        max_q = max(w.q_lens) if w.q_lens else 0
        max_k = max(w.seqlen_k) if w.seqlen_k else 0
        self.pro = ia.prologue_params(
            q=inputs["q"], k=inputs["k"], v=inputs["v"], conv_w_k=inputs["conv_w_k"],
            conv_w_v=inputs["conv_w_v"], q_norm_w=inputs["q_norm_w"], k_norm_w=inputs["k_norm_w"],
            cu_seqlens_q=inputs["cu_seqlens_q"], state_slot=inputs["state_slot"],
            slot_mapping=inputs["slot_mapping"], conv_state_k=inputs["conv_state_k"],
            conv_state_v=inputs["conv_state_v"], q_out=self.q_out, k_cache=inputs["k_cache"],
            v_cache=inputs["v_cache"], max_seqlen_q=max_q, eps=w.eps, dev_status=self.status,
            k_scale=inputs.get("k_scale"), v_scale=inputs.get("v_scale"))
        self.attn = ia.attn_params(
            q=self.q_out, k_cache=inputs["k_cache"], v_cache=inputs["v_cache"],
            cu_seqlens_q=inputs["cu_seqlens_q"], seqlen_k=inputs["seqlen_k"],
            block_table=inputs["block_table"], out=self.out, max_seqlen_q=max_q, max_seqlen_k=max_k,
            r=inputs["r"], P=inputs["P"], rel_extent=w.rel_extent, window=w.window,
            log_scale_base=w.log_scale_base, lse=self.lse, dev_status=self.status,
            k_scale=inputs.get("k_scale"), v_scale=inputs.get("v_scale"))
        self.num_splits = 0
        self.workspace: Optional[torch.Tensor] = None
        self.e4m3 = inputs["k_cache"].dtype == torch.uint8
        if mode == "prefill" and self.e4m3:
            nbytes = ia.inkattn_prefill_workspace_bytes(self.attn)
            self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        if mode == "decode":
            self.num_splits = num_splits if num_splits > 0 else self.heuristic_splits()
            nbytes = ia.inkattn_decode_workspace_bytes(self.attn, self.num_splits)
            if nbytes:
                self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)

    def heuristic_splits(self) -> int:
        sms = torch.cuda.get_device_properties(self.x["q"].device).multi_processor_count
        return ia.inkattn_decode_num_splits(self.attn, sms)

    def run_prologue(self, stream=None):
        ia.inkattn_prologue(self.pro, stream)

    def run_attention(self, stream=None):
        if self.mode == "prefill" and self.e4m3:
            ia.inkattn_prefill_e4m3(self.attn, self.workspace, stream)
        elif self.mode == "prefill":
            ia.inkattn_prefill(self.attn, stream)
        else:
            ia.inkattn_decode(self.attn, self.num_splits, self.workspace, stream)
            ia.inkattn_combine(self.attn, self.num_splits, self.workspace, stream)

    def run(self, stream=None):
        self.run_prologue(stream)
        self.run_attention(stream)

    def launches_per_run(self) -> int:
        n = 2
        if (self.mode == "decode" and self.num_splits > 1) or (self.mode == "prefill" and self.e4m3):
            n += 1
        return n

    def device_status(self) -> int:
        return int(self.status.item())


class OutputConvStep:
    """Buffers + call of the attention-output ShortConv with the residual add and the
    RMSNorm (inkattn_output_conv) over a workload's new tokens.

    `inputs` comes from inputs.make_output_conv_inputs; y stands in for the o_proj
    output.  The conv state in `inputs` is updated in place by every run; h (the new
    residual stream) and out (its RMSNorm) are buffers of this object.
    """

    def __init__(self, w: Workload, inputs: Dict[str, torch.Tensor]):
        self.w, self.x = w, inputs
        dev = inputs["y"].device
        self.h = torch.empty_like(inputs["y"])
        self.out = torch.empty_like(inputs["y"])
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.p = ia.output_conv_params(
            y=inputs["y"], conv_w=inputs["conv_w"], norm_w=inputs["norm_w"],
            cu_seqlens_q=inputs["cu_seqlens_q"], state_slot=inputs["state_slot"],
            conv_state=inputs["conv_state"], residual=inputs["residual"], h_out=self.h, out=self.out,
            max_seqlen_q=max(w.q_lens) if w.q_lens else 0, eps=w.eps, dev_status=self.status)

    def run(self, stream=None):
        ia.inkattn_output_conv(self.p, stream)

    def device_status(self) -> int:
        return int(self.status.item())


class QkvrStep:
    """Buffers + call of the qkvr projections with the prologue fused in
    (inkattn_qkvr_prologue) over a workload's new tokens.

    `inputs` comes from inputs.make_qkvr_inputs.  The conv state is read from
    inputs["conv_state_k"/"conv_state_v"] and the new state written to this object's
    state_k / state_v (in place when `in_place`, allowed when every sequence fits one
    tile); q_out, r_out and, with want_y, y_out (the projections) are buffers of this object;
    the caches in `inputs` receive the new rows.
    """

    def __init__(self, w: Workload, inputs: Dict[str, torch.Tensor], in_place: bool = False,
                 want_y: bool = False):
        self.w, self.x = w, inputs
        dev = inputs["x"].device
        N = w.N_tok
        self.q_out = torch.empty((N, w.Hq, w.head_dim), dtype=torch.bfloat16, device=dev)
        self.r_out = torch.empty((N, w.Hq, w.d_r), dtype=torch.bfloat16, device=dev)
        self.y_out = (torch.empty((N, inputs["w_qkvr"].shape[0]), dtype=torch.bfloat16, device=dev)
                      if want_y else None)
        if in_place:
            self.state_k, self.state_v = inputs["conv_state_k"], inputs["conv_state_v"]
        else:
            self.state_k = torch.empty_like(inputs["conv_state_k"])
            self.state_v = torch.empty_like(inputs["conv_state_v"])
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.p = ia.qkvr_params(
            x=inputs["x"], w=inputs["w_qkvr"], conv_w_k=inputs["conv_w_k"], conv_w_v=inputs["conv_w_v"],
            q_norm_w=inputs["q_norm_w"], k_norm_w=inputs["k_norm_w"], cu_seqlens_q=inputs["cu_seqlens_q"],
            state_slot=inputs["state_slot"], slot_mapping=inputs["slot_mapping"],
            conv_state_k_in=inputs["conv_state_k"], conv_state_v_in=inputs["conv_state_v"],
            conv_state_k_out=self.state_k, conv_state_v_out=self.state_v, q_out=self.q_out,
            r_out=self.r_out, k_cache=inputs["k_cache"], v_cache=inputs["v_cache"],
            max_seqlen_q=max(w.q_lens) if w.q_lens else 0, eps=w.eps, dev_status=self.status,
            k_scale=inputs.get("k_scale"), v_scale=inputs.get("v_scale"), y_out=self.y_out)

    def run(self, stream=None):
        ia.inkattn_qkvr_prologue(self.p, stream)

    def device_status(self) -> int:
        return int(self.status.item())
