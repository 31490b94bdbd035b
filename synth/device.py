"""Put a synthetic workload on the GPU: cache contents, the decode queries and the tokens
appended at every step, generated in place by the GPU twin of synth.gen (or uploaded
from the host generator for small cases). Input generation only."""
from __future__ import annotations

import numpy as np
import torch

from . import gen, gpu
from .workload import HostWorkload


def _bf16(a: np.ndarray, device):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


class DeviceInputs:
    """q [steps][Ly][B][Hq][D], k_new/v_new [steps][Ly][B][Hkv][D] (bf16, device)."""

    def __init__(self, wl: HostWorkload, steps: int, device, on_device: bool = True):
        cfg = wl.cfg
        self.steps = steps
        if on_device:
            self.model = gpu.DeviceModel(wl, device)
            self.q = torch.empty((steps, cfg.n_layers, cfg.batch, cfg.n_q_heads, cfg.head_dim),
                                 dtype=torch.bfloat16, device=device)
            shape = (steps, cfg.n_layers, cfg.batch, cfg.n_kv_heads, cfg.head_dim)
            self.k_new = torch.empty(shape, dtype=torch.bfloat16, device=device)
            self.v_new = torch.empty(shape, dtype=torch.bfloat16, device=device)
            len0 = torch.from_numpy(wl.len0.astype(np.int64)).to(device)
            gpu.fill_queries(wl, self.q, self.model)
            gpu.fill_new_tokens(wl, self.k_new, self.v_new, len0, self.model)
        else:
            self.model = None
            self.q = _bf16(wl.queries(steps), device)
            self.k_new = _bf16(wl.new_tokens("k", steps), device)
            self.v_new = _bf16(wl.new_tokens("v", steps), device)


def fill_state_cache(wl: HostWorkload, state, on_device: bool = True, model=None):
    """Write the prefill rows of every sequence into state.k / state.v."""
    cfg = wl.cfg
    dev = state.k.device
    if on_device:
        model = model or gpu.DeviceModel(wl, dev)
        fill = torch.from_numpy(wl.len0.astype(np.int64)).to(dev)
        owners = gpu.page_owners(wl, dev) if cfg.page_size else None
        gpu.fill_cache(wl, state.k, state.v, fill, model, owners)
    else:
        if cfg.page_size:
            state.k.copy_(_bf16(wl.cache_paged("k"), dev))
            state.v.copy_(_bf16(wl.cache_paged("v"), dev))
        else:
            state.k.copy_(_bf16(wl.cache_contiguous("k", state.capacity), dev))
            state.v.copy_(_bf16(wl.cache_contiguous("v", state.capacity), dev))
    return model


def schedule(wl: HostWorkload, state, steps: int | None = None) -> np.ndarray:
    """Slow flags [steps][B] of the workload's first `steps` decode steps, from the native
    trigger policy: on the boundary masks, or on the generated token streams for a
    token-triggered workload."""
    n = wl.cfg.steps if steps is None else steps
    if wl.cfg.trigger == "tokens":
        return state.schedule_tokens(wl.tokens[:, :n], gen.TRIGGER_TOKENS)
    return state.schedule(wl.masks[:, :n])


def boundary_epochs(wl: HostWorkload, steps: int) -> np.ndarray:
    """Heavy-hitter epoch of every step (uniform boundary mask): boundaries seen before t."""
    m = wl.masks[0][:steps]
    e = np.zeros(steps, dtype=np.int64)
    e[1:] = np.cumsum(m[:-1])
    return e


class DriftingRun:
    """Issues a decode run in segments between boundary steps; before the first step of each
    epoch the drifting heavy-hitter keys are rewritten in place (a harness-side input edit,
    the same one the oracle replays). The run starts by restoring epoch 0, so it can be
    captured once and replayed."""

    def __init__(self, wl: HostWorkload, state, slow, q, k_new, v_new, out, model=None,
                 events=None, **plan_kw):
        cfg = wl.cfg
        self.wl, self.state, self.model = wl, state, model
        steps = slow.shape[0]
        self.ep = boundary_epochs(wl, steps)
        cuts = [t for t in range(1, steps) if self.ep[t] != self.ep[t - 1]] if cfg.drift else []
        bounds = [0] + cuts + [steps]
        self.edits = gpu.drift_edits(wl, state.k.device) if cfg.drift else {}
        self.plans = []
        for a, b in zip(bounds[:-1], bounds[1:]):
            ev = None if events is None else events[2 * a:2 * b]
            self.plans.append((a, state.make_plan(slow, q, k_new, v_new, out, t0=a, t1=b,
                                                  events=ev, **plan_kw)))

    def issue(self, stream=None):
        s = (torch.cuda.current_stream() if stream is None else stream).cuda_stream
        if 0 in self.edits:
            gpu.apply_drift(self.wl, self.state.k, self.edits[0], self.model, s)
        for a, plan in self.plans:
            if a > 0 and int(self.ep[a]) in self.edits:
                gpu.apply_drift(self.wl, self.state.k, self.edits[int(self.ep[a])], self.model, s)
            self.state.run(plan, stream=stream)


def make_state(wl: HostWorkload, device="cuda", on_device: bool = True):
    from sparse_long_context_sfi_gb300.engine import SfiState
    state = SfiState(wl.cfg, wl.len0, device=device, page_table=wl.table, n_pages=wl.n_pages)
    fill_state_cache(wl, state, on_device)
    return state
