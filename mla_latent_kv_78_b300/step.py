"""Device buffers and call order of one MLA decode step.

A step appends this step's n_q new tokens per sequence to the paged latent
cache, absorbs the queries through W^{UK}, runs paged latent attention and
un-absorbs through W^{UV} — four library calls on one stream. PyTorch only
allocates the buffers; every arithmetic step runs in libmla_b300.so.
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import _lib as L


class DecodeStep:
    """Owns the pool, workspace and outputs for a fixed batch shape.

    block_table: int32 [B, max_pages] (page ids); seq_lens: cached lengths
    including this step's n_q tokens; w_uk / w_uv: [H, D, C] act-dtype device
    tensors. All tensors are allocated on ``device``.
    """

    _graph = None
    _graph_events = None

    def __init__(self, cfg: L.mla_config, block_table: torch.Tensor, seq_lens: Sequence[int],
                 n_q: int, num_pages: int, w_uk: torch.Tensor, w_uv: torch.Tensor,
                 num_splits: int = 0, device: str = "cuda"):
        self.cfg = cfg
        self.device = torch.device(device)
        self.n_q = n_q
        self.B = int(block_table.shape[0])
        self.H, self.D, self.C, self.R = cfg.n_heads, cfg.d_head, cfg.d_latent, cfg.d_rope
        self.seq_lens_host = [int(x) for x in seq_lens]
        self.max_seq_len = max(self.seq_lens_host)
        self.num_pages = num_pages
        self.num_splits = num_splits
        act = L.TORCH_ACT[cfg.act_dtype]
        self.act = act
        dev = self.device
        self.block_table = block_table.to(dev, torch.int32).contiguous()
        self.seq_lens = torch.tensor(self.seq_lens_host, dtype=torch.int32, device=dev)
        self.entry_bytes = L.mla_cache_entry_bytes(cfg)
        self.pool = torch.zeros((num_pages, cfg.page_size, self.entry_bytes), dtype=torch.uint8,
                                device=dev)
        self.w_uk = w_uk
        self.w_uv = w_uv
        T = self.B * n_q
        self.T = T
        # positions and page-table rows of this step's new tokens, t = b * n_q + j
        pos = [Lb - n_q + j for Lb in self.seq_lens_host for j in range(n_q)]
        self.step_pos = torch.tensor(pos, dtype=torch.int32, device=dev)
        self.step_seq = torch.arange(self.B, dtype=torch.int32, device=dev).repeat_interleave(n_q)
        self.q_lat = torch.empty((T, self.H, self.C + self.R), dtype=act, device=dev)
        self.o_lat = torch.empty((T, self.H, self.C), dtype=act, device=dev)
        self.lse = torch.empty((T, self.H), dtype=torch.float32, device=dev)
        self.o = torch.empty((T, self.H, self.D), dtype=torch.float32, device=dev)
        ws = L.mla_decode_workspace_size(cfg, self.B, n_q, self.max_seq_len, num_splits)
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)

    # -- cache fill ------------------------------------------------------
    def prefill(self, c_kv: torch.Tensor, k_r: torch.Tensor, seq_idx: torch.Tensor,
                pos: torch.Tensor, stream=None) -> None:
        """Write already-cached tokens (any order) into the pool."""
        L.mla_append_cache(self.cfg, c_kv, k_r, seq_idx, pos, self.block_table, self.pool,
                           self.num_pages, self.dev_status, stream)

    # -- one decode step -------------------------------------------------
    def append(self, c_kv_new, k_r_new, stream=None) -> None:
        L.mla_append_cache(self.cfg, c_kv_new, k_r_new, self.step_seq, self.step_pos,
                           self.block_table, self.pool, self.num_pages, self.dev_status, stream)

    def absorb(self, q_c, q_r, stream=None) -> None:
        L.mla_absorb_q(self.cfg, q_c, q_r, self.step_pos, self.w_uk, self.q_lat, stream)

    def append_absorb(self, c_kv_new, k_r_new, q_c, q_r, stream=None) -> None:
        """append() then absorb() as one library call, the absorption overlapping the append."""
        L.mla_append_absorb(self.cfg, c_kv_new, k_r_new, self.step_seq, self.step_pos,
                            self.block_table, self.pool, q_c, q_r, self.w_uk, self.q_lat,
                            self.num_pages, self.dev_status, stream)

    def decode(self, q_lat: Optional[torch.Tensor] = None, stream=None) -> None:
        L.mla_decode(self.cfg, self.q_lat if q_lat is None else q_lat, self.pool, self.block_table,
                     self.seq_lens, self.n_q, self.max_seq_len, self.o_lat, self.lse,
                     self.workspace, self.num_splits, self.num_pages, self.dev_status, stream)

    def unabsorb(self, stream=None) -> None:
        L.mla_unabsorb(self.cfg, self.o_lat, self.w_uv, self.o, stream)

    def step(self, c_kv_new, k_r_new, q_c, q_r, stream=None) -> torch.Tensor:
        """append + absorb -> decode (+combine) -> unabsorb; returns o [B*n_q, H, D] fp32."""
        self.append_absorb(c_kv_new, k_r_new, q_c, q_r, stream)
        self.decode(None, stream)
        self.unabsorb(stream)
        return self.o

    # -- the step as one CUDA graph ----------------------------------------
    def capture(self, c_kv_new, k_r_new, q_c, q_r, timing: bool = False,
                time_decode: bool = False, branches: bool = False) -> None:
        """Record append + absorb (one mla_append_absorb call) -> decode -> unabsorb over these
        input tensors as one CUDA graph, so a step costs one graph launch instead of several
        host-side library calls. The absorption, decode and unabsorb kernels are programmatic
        launches that set up while their predecessor finishes; the absorption also reads its
        inputs while the append runs. branches=True records separate append and absorb calls as
        parallel branches joined before the decode instead; that measured 1.6 us slower than
        the two separate calls in series (125.5 vs 123.9 us on the V2-shaped benchmark), and the
        single call beats both (116.6 vs 119.8 us in series).

        The graph keeps the inputs' device addresses: write each step's inputs into the same
        tensors (copy_) before replay(). One eager step runs first, outside the capture, so
        the library's one-time per-process set-up never happens inside it. With timing=True
        the graph records events at its start and end (read with step_ms()). time_decode=True
        also records events around mla_decode (decode_ms()); an event between two kernels
        turns their programmatic edge into a full dependency, so that graph is for timing the
        decode alone, not the step.
        """
        dev = self.device
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            self.step(c_kv_new, k_r_new, q_c, q_r)
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize(dev)
        timing = timing or time_decode
        ev = ([torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
              if timing else None)
        graph = torch.cuda.CUDAGraph()
        fork = torch.cuda.Stream(device=dev)
        with torch.cuda.graph(graph):
            main = torch.cuda.current_stream(dev)
            if ev:
                ev[0].record()
            if branches:
                # the cache append and the query absorption touch disjoint buffers: they run
                # side by side, and the decode waits for both
                fork.wait_stream(main)
                with torch.cuda.stream(fork):
                    self.append(c_kv_new, k_r_new)
                self.absorb(q_c, q_r)
                main.wait_stream(fork)
            else:
                self.append_absorb(c_kv_new, k_r_new, q_c, q_r)
            if time_decode:
                ev[1].record()
            self.decode()
            if time_decode:
                ev[2].record()
            self.unabsorb()
            if ev:
                ev[3].record()
        self._graph = graph
        self._graph_events = ev

    def replay(self) -> torch.Tensor:
        """Launch the captured step on the current stream; returns o."""
        self._graph.replay()
        return self.o

    def step_ms(self) -> float:
        e = self._graph_events
        return e[0].elapsed_time(e[3])

    def decode_ms(self) -> float:
        e = self._graph_events
        return e[1].elapsed_time(e[2])

    def status(self) -> int:
        return int(self.dev_status.item())
