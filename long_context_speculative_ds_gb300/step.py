"""One verify step through the C ABI: per-layer tree-verify attention with
chunk salience summed over layers, then top-k chunk gather into the compact
draft cache, then tree acceptance, then (optionally) the commit of the
accepted path into every layer's cache.

`VerifyStep` owns the device buffers of a step (outputs and workspaces) for
fixed sizes; every computation is a call into the library.  Inputs are passed
in as device tensors (already resident) or copied in from pinned host
tensors by `upload` for end-to-end timing.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence

import torch

from . import binding as B


def max_chunks_for(max_pages: int, page_size: int, chunk_size: int) -> int:
    return -(-(max_pages * page_size) // chunk_size)


@dataclass
class StepInputs:
    """Device (or pinned host) tensors of one step."""
    page_table: torch.Tensor        # [B, max_pages] int32
    ctx_lens: torch.Tensor          # [B] int32
    tree_offsets: torch.Tensor      # [B+1] int32
    parents: torch.Tensor           # [n_nodes] int32
    q: List[torch.Tensor]           # per layer [n_nodes, H_q, D] bf16
    k_cache: List[torch.Tensor]     # per layer paged bf16
    v_cache: List[torch.Tensor]
    src_k: torch.Tensor             # gather source cache
    src_v: torch.Tensor
    target_logits: torch.Tensor     # [n_nodes, V] fp32
    draft_logits: Optional[torch.Tensor]
    draft_tokens: torch.Tensor      # [n_nodes] int32
    uniforms: Optional[torch.Tensor]


class VerifyStep:
    def __init__(self, inp: StepInputs, *, chunk_size: int, top_k: int,
                 window: int, accept_mode: str, kv_layout: str = "NHD",
                 out_dtype: torch.dtype = torch.bfloat16, num_sms: int = 0,
                 device: str = "cuda", with_commit: bool = False,
                 rope_base: float = 0.0):
        self.inp = inp
        self.chunk_size, self.top_k, self.window = chunk_size, top_k, window
        self.accept_mode = accept_mode
        self.kv_layout = kv_layout
        self.layers = len(inp.q)
        bsz, max_pages = inp.page_table.shape
        k0 = inp.k_cache[0]
        page_size = k0.shape[1] if kv_layout == "NHD" else k0.shape[2]
        kv_heads = k0.shape[2] if kv_layout == "NHD" else k0.shape[1]
        head_dim = k0.shape[3]
        n_nodes, num_q_heads, _ = inp.q[0].shape
        self.max_chunks = max_chunks_for(max_pages, page_size, chunk_size)
        dev = torch.device(device)
        self.out = [torch.empty(n_nodes, num_q_heads, head_dim, dtype=out_dtype,
                                device=dev) for _ in range(self.layers)]
        self.scores = torch.zeros(bsz, self.max_chunks, dtype=torch.float32,
                                  device=dev)
        a = B.verify_args(inp.q[0], k0, inp.v_cache[0], inp.page_table,
                          inp.ctx_lens, inp.tree_offsets, inp.parents,
                          chunk_size=chunk_size, out=self.out[0],
                          chunk_scores=self.scores, kv_layout=kv_layout,
                          num_sms=num_sms)
        self.ws_verify = torch.zeros(B.ds_verify_attn_workspace_size(a),
                                     dtype=torch.uint8, device=dev)
        self.verify_args = []
        for l in range(self.layers):
            self.verify_args.append(B.verify_args(
                inp.q[l], inp.k_cache[l], inp.v_cache[l], inp.page_table,
                inp.ctx_lens, inp.tree_offsets, inp.parents,
                chunk_size=chunk_size, out=self.out[l],
                chunk_scores=self.scores, workspace=self.ws_verify,
                kv_layout=kv_layout, accumulate=l > 0, num_sms=num_sms))
        cap = top_k * chunk_size + window
        self.capacity = cap
        self.out_k = torch.empty(bsz, cap, kv_heads, head_dim,
                                 dtype=torch.bfloat16, device=dev)
        self.out_v = torch.empty_like(self.out_k)
        self.out_positions = torch.empty(bsz, cap, dtype=torch.int32, device=dev)
        self.out_len = torch.empty(bsz, dtype=torch.int32, device=dev)
        self.out_chunk_ids = torch.empty(bsz, max(top_k, 1), dtype=torch.int32,
                                         device=dev)
        self.ws_gather = torch.zeros(256, dtype=torch.uint8, device=dev)
        self.gather_args = B.gather_args(
            self.scores, inp.ctx_lens, inp.src_k, inp.src_v, inp.page_table,
            chunk_size=chunk_size, top_k=top_k, window=window,
            out_k=self.out_k, out_v=self.out_v,
            out_positions=self.out_positions, out_len=self.out_len,
            out_chunk_ids=self.out_chunk_ids, workspace=self.ws_gather,
            kv_layout=kv_layout, rope_base=rope_base)
        self.out_path = torch.empty(bsz, B.DS_MAX_TREE_NODES, dtype=torch.int32,
                                    device=dev)
        self.out_n = torch.empty(bsz, dtype=torch.int32, device=dev)
        self.out_bonus = torch.empty(bsz, dtype=torch.int32, device=dev)
        aa = B.accept_args(accept_mode, inp.target_logits, inp.draft_tokens,
                           inp.parents, inp.tree_offsets,
                           out_path=self.out_path, out_n_accepted=self.out_n,
                           out_bonus=self.out_bonus,
                           draft_logits=inp.draft_logits,
                           uniforms=inp.uniforms)
        self.ws_accept = torch.zeros(B.ds_accept_workspace_size(aa),
                                     dtype=torch.uint8, device=dev)
        self.accept_args = B.accept_args(
            accept_mode, inp.target_logits, inp.draft_tokens, inp.parents,
            inp.tree_offsets, out_path=self.out_path,
            out_n_accepted=self.out_n, out_bonus=self.out_bonus,
            draft_logits=inp.draft_logits, uniforms=inp.uniforms,
            workspace=self.ws_accept)
        self.with_commit = with_commit
        self.new_ctx_lens = torch.empty(bsz, dtype=torch.int32, device=dev)
        self.ws_commit = torch.zeros(256, dtype=torch.uint8, device=dev)
        if with_commit:
            self.commit_args = B.commit_args(
                inp.k_cache, inp.v_cache, inp.page_table, inp.ctx_lens,
                inp.tree_offsets, self.out_path, self.out_n,
                new_ctx_lens=self.new_ctx_lens, workspace=self.ws_commit,
                kv_layout=kv_layout)
        for ws in (self.ws_verify, self.ws_gather, self.ws_accept, self.ws_commit):
            B.ds_workspace_init(ws)

    # -- the step ----------------------------------------------------------
    def verify_layer(self, l: int, stream=None):
        B.ds_verify_attn(self.verify_args[l], stream)

    def gather(self, stream=None):
        B.ds_chunk_topk_gather(self.gather_args, stream)

    def accept(self, stream=None):
        B.ds_accept(self.accept_args, stream)

    def commit(self, stream=None):
        B.ds_kv_commit(self.commit_args, stream)

    def run(self, stream=None):
        for l in range(self.layers):
            self.verify_layer(l, stream)
        self.gather(stream)
        self.accept(stream)
        if self.with_commit:
            self.commit(stream)

    def launches_per_step(self) -> int:
        """Kernel launches of one step: 2 per layer (split pass, finish),
        2 for top-k + gather, 2 for acceptance, 1 for the commit."""
        return self.layers * 2 + 2 + 2 + (1 if self.with_commit else 0)

    def device_status(self) -> int:
        s = 0
        for ws in (self.ws_verify, self.ws_gather, self.ws_accept, self.ws_commit):
            s |= B.ds_device_status(ws)
        return s

    # -- end-to-end helpers ------------------------------------------------
    def upload(self, host: "StepInputs", stream=None):
        """Copy a step's per-step inputs from pinned host tensors into the
        step's device tensors (asynchronously on the current stream)."""
        d = self.inp
        pairs = [(d.page_table, host.page_table), (d.ctx_lens, host.ctx_lens),
                 (d.tree_offsets, host.tree_offsets), (d.parents, host.parents),
                 (d.target_logits, host.target_logits),
                 (d.draft_tokens, host.draft_tokens)]
        if d.draft_logits is not None:
            pairs.append((d.draft_logits, host.draft_logits))
        if d.uniforms is not None:
            pairs.append((d.uniforms, host.uniforms))
        for l in range(self.layers):
            pairs.append((d.q[l], host.q[l]))
        n = 0
        for dst, src in pairs:
            dst.copy_(src, non_blocking=True)
            n += src.numel() * src.element_size()
        return n

    def run_from_host(self, host: "StepInputs", host_out: dict):
        """One step end to end from pinned host inputs, with the copies on a
        side stream: the tree, then each layer's Q, then the logits, each
        group behind an event that only the kernels reading it wait on, so
        the copies of later layers and of the logits overlap the verify of
        earlier layers.  The side stream first waits for the current stream
        (the previous step's kernels may still read these buffers).

        A wait on an event between two kernels of the step breaks their
        dependent launch, so there are few: layer 0 waits for the tree and
        its Q, layer 1 for its Q, layer 2 for every remaining layer's Q (a
        Q copy takes a few microseconds, a layer's verify over a hundred, so
        they are done by then), and acceptance for the logits.
        Returns (host-to-device bytes, device-to-host bytes)."""
        comp = torch.cuda.current_stream()
        if getattr(self, "_copy_stream", None) is None:
            self._copy_stream = torch.cuda.Stream()
            self._ev_tree = torch.cuda.Event()
            self._ev_q = [torch.cuda.Event() for _ in range(3)]
            self._ev_acc = torch.cuda.Event()
        cp = self._copy_stream
        cp.wait_stream(comp)
        d = self.inp
        n = 0

        def put(dst, src):
            nonlocal n
            dst.copy_(src, non_blocking=True)
            n += src.numel() * src.element_size()

        with torch.cuda.stream(cp):
            for dst, src in ((d.page_table, host.page_table), (d.ctx_lens, host.ctx_lens),
                             (d.tree_offsets, host.tree_offsets), (d.parents, host.parents)):
                put(dst, src)
            self._ev_tree.record(cp)
            for l in range(self.layers):
                put(d.q[l], host.q[l])
                if l < 2 or l == self.layers - 1:
                    self._ev_q[min(l, 2)].record(cp)
            put(d.target_logits, host.target_logits)
            put(d.draft_tokens, host.draft_tokens)
            if d.draft_logits is not None:
                put(d.draft_logits, host.draft_logits)
            if d.uniforms is not None:
                put(d.uniforms, host.uniforms)
            self._ev_acc.record(cp)
        comp.wait_event(self._ev_tree)
        for l in range(self.layers):
            if l <= 2:
                comp.wait_event(self._ev_q[l])
            self.verify_layer(l)
        self.gather()
        comp.wait_event(self._ev_acc)
        self.accept()
        if self.with_commit:
            self.commit()
        return n, self.download(host_out)

    def capture_from_host(self, host: "StepInputs", host_out: dict):
        """Capture one end-to-end step (`run_from_host`: the copies in, every
        kernel, the copies out) as a CUDA graph; `replay` then runs the whole
        step again with one launch, from whatever the pinned host buffers
        hold at that time.  Buffers, sizes and the library's arguments are
        those of the capture.  Call it after one eager `run_from_host`: the
        library sets function attributes on first use, which a stream
        capture does not allow.  Returns what `run_from_host` returns."""
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, capture_error_mode="thread_local"):
            self._graph_bytes = self.run_from_host(host, host_out)
        self._graph = graph
        return self._graph_bytes

    def replay(self):
        """One end-to-end step through the captured graph (asynchronous on
        the current stream).  Returns (host-to-device, device-to-host) bytes."""
        self._graph.replay()
        return self._graph_bytes

    def download(self, host_out: dict):
        """Copy the step's small results (accepted path, count, bonus, chosen
        chunks, compact length) to pinned host tensors."""
        n = 0
        for name in ("out_path", "out_n", "out_bonus", "out_chunk_ids",
                     "out_len"):
            src = getattr(self, name)
            host_out[name].copy_(src, non_blocking=True)
            n += src.numel() * src.element_size()
        return n
