"""Device state of one SFI decode workload and the calls that step it.

`SfiState` owns (through PyTorch allocations) the KV cache, the packed sparse memory, the
evidence buffer and the workspace, and builds the C descriptors. Stepping goes through the
C ABI only: `step()` issues the per-step calls, `run()` hands a whole decode run to the
native driver `sfi_decode_run` (capturable in a CUDA graph).
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import torch

from . import (SfiBudget, SfiDecodePlan, SfiKvCache, SfiSparseMem, sfi_append_kv, sfi_compact,
               sfi_decode_run, sfi_dense_decode_attn, sfi_schedule, sfi_schedule_tokens,
               sfi_select, sfi_fast_decode_step, sfi_sparse_decode_attn, sfi_workspace_bytes,
               sfi_workspace_init)


class SfiState:
    def __init__(self, cfg, len0, device="cuda", page_table=None, n_pages=0, capacity=None):
        self.cfg = cfg
        self.device = torch.device(device)
        B, Ly, Hkv, Hq, D = cfg.batch, cfg.n_layers, cfg.n_kv_heads, cfg.n_q_heads, cfg.head_dim
        self.len0 = np.asarray(len0, dtype=np.int64)
        self.capacity = capacity or int(self.len0.max()) + cfg.steps
        bf = torch.bfloat16
        if cfg.page_size:
            pt = np.asarray(page_table, dtype=np.int32)
            self.page_table = torch.from_numpy(pt).to(self.device)
            self.n_pages = int(n_pages)
            self.max_pages = int(pt.shape[1])
            self.capacity = self.max_pages * cfg.page_size
            shape = (Ly, self.n_pages, Hkv, cfg.page_size, D)
        else:
            self.page_table = None
            self.n_pages = 0
            self.max_pages = 0
            shape = (Ly, B, Hkv, self.capacity, D)
        self.k = torch.zeros(shape, dtype=bf, device=self.device)
        self.v = torch.zeros(shape, dtype=bf, device=self.device)
        self.seq_len = torch.from_numpy(self.len0.astype(np.int32)).to(self.device)
        self.err = torch.zeros(4, dtype=torch.int32, device=self.device)
        U = Ly * B * Hkv
        self.n_units = U
        comp = cfg.n_sink + cfg.n_select
        self.kc = torch.zeros((Ly, B, Hkv, comp, D), dtype=bf, device=self.device)
        self.vc = torch.zeros((Ly, B, Hkv, comp, D), dtype=bf, device=self.device)
        self.sel_idx = torch.zeros((U, max(1, cfg.n_select)), dtype=torch.int32, device=self.device)
        self.sel_cnt = torch.zeros(U, dtype=torch.int32, device=self.device)
        self.rows = torch.zeros(U, dtype=torch.int32, device=self.device)
        self.scores = torch.zeros((U, self.capacity), dtype=torch.float32, device=self.device)
        self.kv = SfiKvCache(
            n_layers=Ly, batch=B, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, capacity=self.capacity,
            page_size=cfg.page_size, n_pages=self.n_pages, max_pages_per_seq=self.max_pages,
            max_len=int(self.len0.max()), k=self.k.data_ptr(), v=self.v.data_ptr(),
            page_table=None if self.page_table is None else self.page_table.data_ptr(),
            seq_len=self.seq_len.data_ptr(), err=self.err.data_ptr())
        self.budget = SfiBudget(n_sink=cfg.n_sink, n_window=cfg.n_window, n_select=cfg.n_select,
                                prior_tau=cfg.prior_tau, lambda_=cfg.lam)
        self.mem = SfiSparseMem(kc=self.kc.data_ptr(), vc=self.vc.data_ptr(),
                                sel_idx=self.sel_idx.data_ptr(), sel_cnt=self.sel_cnt.data_ptr(),
                                rows=self.rows.data_ptr())
        self.ws_bytes = sfi_workspace_bytes(self.kv, self.budget)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        sfi_workspace_init(self.ws, self.ws_bytes)
        self.t = 0

    # -- host bookkeeping -------------------------------------------------------------------
    def reset_lengths(self):
        self.seq_len.copy_(torch.from_numpy(self.len0.astype(np.int32)))
        self.t = 0

    def schedule(self, masks: np.ndarray) -> np.ndarray:
        """Slow flags [steps][B] from per-sequence boundary masks [B][steps]."""
        return np.stack([sfi_schedule(masks[b], self.cfg.t_max) for b in range(self.cfg.batch)], 1)

    def schedule_tokens(self, tokens: np.ndarray, trigger_ids) -> np.ndarray:
        """Slow flags [steps][B] from per-sequence generated token ids [B][steps]: a slow step
        follows a trigger token (or T_max steps without one)."""
        return np.stack([sfi_schedule_tokens(tokens[b], trigger_ids, self.cfg.t_max)
                         for b in range(self.cfg.batch)], 1)

    # -- one decode step through the individual calls -----------------------------------------
    def step(self, q, k_new, v_new, slow_b: np.ndarray, out, out_fp32=True, stream=None,
             fused=True):
        """q [Ly][B][Hq][D] bf16, k_new/v_new [Ly][B][Hkv][D] bf16 (device); slow_b [B] bool.
        fused: the fast sequences' append runs inside sfi_fast_decode_step (as in the native
        driver); otherwise every row is appended first and the fast step is
        sfi_sparse_decode_attn."""
        kv = self.kv
        bound = int(self.len0.max()) + self.t
        slow_b = np.asarray(slow_b, bool)
        mixed = slow_b.any() and not slow_b.all()
        if mixed:
            m = torch.from_numpy(np.stack([slow_b, ~slow_b]).astype(np.uint8)).to(self.device)
            a_slow, a_fast = m[0], m[1]
        else:
            a_slow = a_fast = None
        kv.max_len = bound
        if not fused:
            sfi_append_kv(kv, k_new, v_new, stream=stream)
        elif slow_b.any():
            sfi_append_kv(kv, k_new, v_new, active=a_slow, stream=stream)
        kv.max_len = bound + 1
        if slow_b.any():
            sfi_dense_decode_attn(kv, q, out, out_fp32, self.scores, self.ws, self.ws_bytes,
                                  active=a_slow, stream=stream)
            sfi_select(kv, self.scores, self.budget, self.mem, active=a_slow, stream=stream)
            sfi_compact(kv, self.budget, self.mem, active=a_slow, stream=stream)
        if not slow_b.all():
            if fused:
                kv.max_len = bound
                sfi_fast_decode_step(kv, self.mem, self.budget, k_new, v_new, q, out, out_fp32,
                                     self.ws, self.ws_bytes, active=a_fast, stream=stream)
                kv.max_len = bound + 1
            else:
                sfi_sparse_decode_attn(kv, self.mem, self.budget, q, out, out_fp32, self.ws,
                                       self.ws_bytes, active=a_fast, stream=stream)
        self.t += 1
        return mixed and (a_slow, a_fast)

    # -- a whole run through the native driver --------------------------------------------------
    def side_stream(self, priority=0):
        """The layer-wise pipeline's side stream and its fork and join events (created once;
        the events are recorded once here so that their driver objects exist before any
        stream capture)."""
        if getattr(self, "_side", None) is None:
            side = torch.cuda.Stream(device=self.device, priority=priority)
            fork, join = torch.cuda.Event(), torch.cuda.Event()
            fork.record()
            join.record()
            torch.cuda.synchronize(self.device)
            self._side = (side, fork, join)
        return self._side

    def make_plan(self, slow: np.ndarray, q, k_new, v_new, out, out_fp32=True, out_per_step=True,
                  dense_only=False, events=None, t0=0, t1=None, pipeline=False, pipeline_group=0,
                  concurrent=None):
        """slow: uint8 [steps][B]; q/k_new/v_new/out: device tensors with a leading step axis.
        events: optional list of 2 * (t1 - t0) torch.cuda.Event(enable_timing=True) or None,
        recorded before (2 t) and after (2 t + 1) step t's attention kernel (None: not
        recorded). [t0, t1): the steps this plan covers (a run can be issued as several
        consecutive plans). pipeline: run slow steps group of layers by group, with the
        Selector and compaction of each group on a side stream beside the next group's
        attention; pipeline_group: layers per group (0: about a quarter of the layers).
        concurrent: on steps that mix slow and fast sequences, the fast sequences' fused fast
        step runs on a side stream beside the slow sequences' chain (not with pipeline; the
        results are the same bits); None: on when the plan has such a step."""
        t1 = slow.shape[0] if t1 is None else t1
        q, k_new, v_new = q[t0:t1], k_new[t0:t1], v_new[t0:t1]
        if out_per_step:
            out = out[t0:t1]
        slow = np.ascontiguousarray(slow[t0:t1], dtype=np.uint8)
        steps = slow.shape[0]
        mixed = np.array([(r.any() and not r.all()) for r in slow])
        masks = None
        if concurrent is None:
            concurrent = bool(mixed.any()) and not pipeline and not dense_only
        if mixed.any():
            m = np.stack([slow, 1 - slow], axis=1).astype(np.uint8)
            masks = torch.from_numpy(m).to(self.device)
        plan = SfiDecodePlan(
            n_steps=steps, slow=slow.ctypes.data, q=q.data_ptr(), k_new=k_new.data_ptr(),
            v_new=v_new.data_ptr(), out=out.data_ptr(), out_fp32=1 if out_fp32 else 0,
            out_per_step=1 if out_per_step else 0, scores_f=self.scores.data_ptr(),
            masks=None if masks is None else masks.data_ptr(),
            len_start=int(self.len0.max()) + t0, dense_only=1 if dense_only else 0)
        if pipeline or concurrent:
            side, fork, join = self.side_stream()
            plan.side_stream, plan.fork_event, plan.join_event = (side.cuda_stream, fork.cuda_event,
                                                                  join.cuda_event)
            plan.pipeline_group = int(pipeline_group)
            plan.concurrent_fast = 1 if concurrent and not pipeline else 0
        ev_arr = None
        if events is not None:
            assert len(events) == 2 * steps
            for e in events:          # make sure the driver-level event objects exist
                if e is not None:
                    e.record()
            torch.cuda.synchronize()
            ev_arr = (C.c_void_p * (2 * steps))(*[None if e is None else e.cuda_event
                                                  for e in events])
            plan.events = C.cast(ev_arr, C.c_void_p)
        plan._keep = (slow, masks, q, k_new, v_new, out, ev_arr, events)
        return plan

    def run(self, plan: SfiDecodePlan, stream=None):
        sfi_decode_run(self.kv, self.budget, self.mem, plan, self.ws, self.ws_bytes, stream=stream)
