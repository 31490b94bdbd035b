"""Seeded, counter-based synthetic inputs for the SFI decode-attention workloads.

This module is shared by the oracle and by the CUDA path's tests and benchmark. It holds
none of the method's arithmetic: it only turns (seed, stream, layer, sequence, head,
position, dim) coordinates into bf16 bit patterns, host tables and masks. The GPU twin
in ``synth/csrc/synth_gen.cu`` evaluates the same formulas bit for bit, so large KV
caches can be produced on the device while the oracle regenerates any slice on the host.

Generator definition (both twins):
  * counter  c = d | pos<<8 | head<<32 | b<<38 | layer<<46 | stream<<54   (uint64)
  * hash     h = mix(key + (c + 1) * GAMMA), mix = the SplitMix64 output function
               (Steele, Lea, Flood, "Fast splittable pseudorandom number generators",
               OOPSLA 2014): z ^= z>>30; z *= M1; z ^= z>>27; z *= M2; z ^= z>>31.
  * normal   Irwin-Hall of the four 16-bit fields u0..u3 of h:
               x = fl32(fl32(u0+u1+u2+u3 - 131070) * 2^-16) * fl32(sqrt(3))  (one RNE multiply)
             mean 0, variance 1 - 2^-32.
  * bf16     round-to-nearest-even of the fp32 value.
"""
from __future__ import annotations

import math

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
M1 = np.uint64(0xBF58476D1CE4E5B9)
M2 = np.uint64(0x94D049BB133111EB)

# Streams: independent sub-sequences of the hash.
STREAM_K, STREAM_V, STREAM_Q, STREAM_ZIPF, STREAM_DIR, STREAM_HH, STREAM_PAGE, STREAM_LEN, \
    STREAM_MASK, STREAM_DRIFT = range(10)

SQRT3_F32 = np.float32(math.sqrt(3.0))
INV_2_16 = np.float32(2.0 ** -16)

ZIPF_EXPONENT = 1.1
ZIPF_KMAX = 4096          # draws beyond the table get boost 1
HEAVY_HITTERS = 32        # planted heavy-hitter keys per (layer, sequence, kv head)


def key_from_seed(seed: int) -> np.uint64:
    """64-bit generator key for an integer seed (the seed itself pushed through the mix)."""
    return mix64(np.uint64(0), np.array([seed], dtype=np.uint64))[0]


def counter(stream, layer, b, head, pos, d) -> np.ndarray:
    """Pack coordinates into the 64-bit counter (broadcasting numpy integer arrays)."""
    u = lambda x: np.asarray(x).astype(np.uint64)
    return (u(d) | (u(pos) << np.uint64(8)) | (u(head) << np.uint64(32)) | (u(b) << np.uint64(38))
            | (u(layer) << np.uint64(46)) | (u(stream) << np.uint64(54)))


def mix64(key, ctr) -> np.ndarray:
    """SplitMix64 output function applied to key + (ctr + 1) * GAMMA (all mod 2^64)."""
    with np.errstate(over="ignore"):
        z = np.asarray(key, dtype=np.uint64) + (np.asarray(ctr, dtype=np.uint64) + np.uint64(1)) * GAMMA
        z = (z ^ (z >> np.uint64(30))) * M1
        z = (z ^ (z >> np.uint64(27))) * M2
        return z ^ (z >> np.uint64(31))


def hash_at(key, stream, layer, b, head, pos, d) -> np.ndarray:
    return mix64(key, counter(stream, layer, b, head, pos, d))


def normal_f32(h: np.ndarray) -> np.ndarray:
    """Approximately N(0,1) fp32 from one 64-bit hash (Irwin-Hall of four 16-bit fields)."""
    m = np.uint64(0xFFFF)
    s = ((h & m) + ((h >> np.uint64(16)) & m) + ((h >> np.uint64(32)) & m)
         + ((h >> np.uint64(48)) & m)).astype(np.int64) - 131070
    x = s.astype(np.float32) * INV_2_16          # exact: |s| < 2^24, power-of-two scale
    return (x * SQRT3_F32).astype(np.float32)    # one RNE fp32 multiply


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = (u & np.uint64(0x7FFFFFFF)) > np.uint64(0x7F800000)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    r = np.where(nan, np.uint64(0x7FC0), r)
    return r.astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------------------------------
# Key-norm models
# ----------------------------------------------------------------------------------------

def zipf_tables():
    """Inverse-CDF table for X ~ Zipf(1.1) on {1, 2, ...} and the boost 1 + 3 X^-1.1.

    thresholds[k-1] = floor(P(X <= k) * 2^32) for k = 1..ZIPF_KMAX (uint32);
    X = min{k : u32 < thresholds[k-1]}, else ZIPF_KMAX + 1.
    boosts[k-1] = fl32(1 + 3 k^-1.1) for k <= ZIPF_KMAX, boosts[ZIPF_KMAX] = 1.
    """
    from scipy.special import zeta
    k = np.arange(1, ZIPF_KMAX + 1, dtype=np.float64)
    w = k ** (-ZIPF_EXPONENT)
    cdf = np.cumsum(w) / zeta(ZIPF_EXPONENT)
    thr = np.minimum(np.floor(cdf * 2.0 ** 32), 2.0 ** 32 - 1).astype(np.uint64).astype(np.uint32)
    boosts = np.empty(ZIPF_KMAX + 1, dtype=np.float32)
    boosts[:ZIPF_KMAX] = (1.0 + 3.0 * w).astype(np.float32)
    boosts[ZIPF_KMAX] = np.float32(1.0)
    return thr, boosts


_ZIPF = None


def _zipf():
    global _ZIPF
    if _ZIPF is None:
        _ZIPF = zipf_tables()
    return _ZIPF


def zipf_boost(key, layer, b, head, pos) -> np.ndarray:
    """Per-position key-norm boost (fp32) for the Zipf key model."""
    thr, boosts = _zipf()
    u = (hash_at(key, STREAM_ZIPF, layer, b, head, pos, 0) >> np.uint64(32)).astype(np.uint32)
    x_index = np.searchsorted(thr, u, side="right")    # = X - 1, or ZIPF_KMAX when beyond
    return boosts[x_index]


def hh_direction(key, n_layers: int, n_kv_heads: int, head_dim: int):
    """Unit query direction per (layer, kv head) for the heavy-hitter key model.

    Returns (qa, ka): fp32 [Ly][Hkv][D] tables with qa = fl32(a u), ka = fl32(4 a u),
    a = sqrt(D)/2, u the normalised Gaussian direction (normalised in double)."""
    lay = np.arange(n_layers)[:, None, None]
    hd = np.arange(n_kv_heads)[None, :, None]
    d = np.arange(head_dim)[None, None, :]
    g = normal_f32(hash_at(key, STREAM_DIR, lay, 0, hd, 0, d)).astype(np.float64)
    u = g / np.sqrt((g * g).sum(axis=-1, keepdims=True))
    a = math.sqrt(head_dim) / 2.0
    return (a * u).astype(np.float32), (4.0 * a * u).astype(np.float32)


def _draw_distinct(key, stream, layer, b, head, base, n, ctx, taken):
    """n distinct positions in [0, ctx) not in `taken`, by rejection: candidate i is
    hash(stream, layer, b, head, base + i) mod ctx (uniform without replacement)."""
    out = []
    i = 0
    while len(out) < n:
        p = int(hash_at(key, stream, layer, b, head, np.array([base + i]), 0)[0] % np.uint64(ctx))
        i += 1
        if p not in taken:
            taken.add(p)
            out.append(p)
    return out


def hh_epochs(key, layer: int, b: int, head: int, ctx: int, n_epochs: int,
              count: int = HEAVY_HITTERS, drift_frac: float = 0.1):
    """Heavy-hitter position sets (sorted) of one (layer, sequence, kv head) for epochs
    0 .. n_epochs-1, in [0, ctx).

    Epoch 0: `count` positions uniform without replacement (rejection on the hash). Each
    later epoch re-seeds round(drift_frac * count) of them: the ones with the smallest
    drift hash are dropped and as many new positions, not already in the set, are drawn
    from that epoch's own stream."""
    cur = sorted(_draw_distinct(key, STREAM_HH, layer, b, head, 0, count, ctx, set()))
    out = [np.array(cur, dtype=np.int64)]
    n_move = int(round(drift_frac * count))
    for e in range(1, n_epochs):
        dh = hash_at(key, STREAM_DRIFT, layer, b, head, np.array(cur), 2 * e)
        drop = set(np.array(cur)[np.argsort(dh, kind="stable")[:n_move]].tolist())
        keep = [p for p in cur if p not in drop]
        new = _draw_distinct(key, STREAM_DRIFT, layer, b, head, (2 * e + 1) << 12, n_move, ctx,
                             set(cur))
        cur = sorted(keep + new)
        out.append(np.array(cur, dtype=np.int64))
    return out


def hh_positions(key, layer: int, b: int, head: int, ctx: int, epoch: int = 0,
                 count: int = HEAVY_HITTERS, drift_frac: float = 0.1) -> np.ndarray:
    """Heavy-hitter positions of one unit at one epoch (see hh_epochs)."""
    return hh_epochs(key, layer, b, head, ctx, epoch + 1, count, drift_frac)[epoch]


def hh_bitmap(positions_per_unit, cap: int) -> np.ndarray:
    """uint32 bitmap [U][ceil(cap/32)] with bit p set for each heavy-hitter position p."""
    words = (cap + 31) // 32
    bm = np.zeros((len(positions_per_unit), words), dtype=np.uint32)
    for u, ps in enumerate(positions_per_unit):
        for p in ps:
            bm[u, p >> 5] |= np.uint32(1) << np.uint32(p & 31)
    return bm


# ----------------------------------------------------------------------------------------
# Tensor content
# ----------------------------------------------------------------------------------------

def kv_rows(key, which: str, layer: int, b: int, head: int, pos: np.ndarray, head_dim: int,
            model: str, ka_row=None, hh_mask=None) -> np.ndarray:
    """bf16 bits [len(pos)][D] of the K ('k') or V ('v') rows at the given positions.

    model 'plain': N(0,1).  model 'zipf': keys scaled by the Zipf boost of their position.
    model 'hh': keys at heavy-hitter positions (hh_mask True) get ka_row added."""
    pos = np.asarray(pos, dtype=np.int64)
    stream = STREAM_K if which == "k" else STREAM_V
    d = np.arange(head_dim)[None, :]
    x = normal_f32(hash_at(key, stream, layer, b, head, pos[:, None], d))
    if which == "k" and model == "zipf":
        x = (x * zipf_boost(key, layer, b, head, pos)[:, None]).astype(np.float32)
    elif which == "k" and model == "hh" and hh_mask is not None and np.any(hh_mask):
        x = np.where(hh_mask[:, None], (x + ka_row[None, :]).astype(np.float32), x)
    return f32_to_bf16(x)


def q_rows(key, step: int, layer: int, b: int, n_q_heads: int, head_dim: int, qa=None,
           group: int = 1) -> np.ndarray:
    """bf16 bits [Hq][D] of the decode query at `step`; qa (optional, [Hkv][D]) is added
    to each head of kv group h // group (heavy-hitter model)."""
    h = np.arange(n_q_heads)[:, None]
    d = np.arange(head_dim)[None, :]
    x = normal_f32(hash_at(key, STREAM_Q, layer, b, h, step, d))
    if qa is not None:
        x = (x + qa[np.arange(n_q_heads) // group]).astype(np.float32)
    return f32_to_bf16(x)


# ----------------------------------------------------------------------------------------
# Host-only data: lengths, masks, page tables
# ----------------------------------------------------------------------------------------

def uniform01(key, stream, b, idx) -> np.ndarray:
    """Doubles in (0, 1) from the top 53 bits of the hash."""
    h = hash_at(key, stream, 0, b, 0, idx, 0)
    return ((h >> np.uint64(11)).astype(np.float64) + 0.5) * 2.0 ** -53


def ragged_lengths(key, batch: int, lo: int, hi: int) -> np.ndarray:
    """Per-sequence prefill lengths, uniform on the integers [lo, hi]."""
    u = uniform01(key, STREAM_LEN, np.arange(batch), 0)
    return (lo + np.floor(u * (hi - lo + 1))).astype(np.int64)


def boundary_mask(key, steps: int, kind: str, param: float, b: int = 0) -> np.ndarray:
    """uint8 [steps]; mask[t] = 1 marks token t as a span boundary (step t+1 is slow).

    'periodic', p: mask[t] = 1 iff (t + 1) % p == 0.
    'geometric', mean: gaps g >= 1 ~ Geometric(1/mean) on {1, 2, ...} drawn by inverse CDF,
    boundaries at the running sums minus one."""
    m = np.zeros(steps, dtype=np.uint8)
    if kind == "periodic":
        p = int(param)
        m[(np.arange(steps) + 1) % p == 0] = 1
        return m
    p = 1.0 / float(param)
    t, i = -1, 0
    while True:
        u = uniform01(key, STREAM_MASK, b, i)
        g = 1 + int(math.floor(math.log(float(u)) / math.log1p(-p)))
        t += g
        i += 1
        if t >= steps:
            return m
        m[t] = 1


TRIGGER_TOKENS = (13, 30, 0, 198)   # synthetic ids standing for ".", "?", "!" and newline


def token_stream(key, steps: int, vocab: int = 32000, mean_span: float = 18.0, b: int = 0,
                 trigger_ids=TRIGGER_TOKENS) -> np.ndarray:
    """int32 [steps] synthetic generated tokens: each token is a trigger id with probability
    1/mean_span (which one: uniform), otherwise a uniform non-trigger id."""
    u = uniform01(key, STREAM_MASK, b, np.arange(steps) + (1 << 20))
    h = hash_at(key, STREAM_MASK, 1, b, 0, np.arange(steps), 1)
    trig = np.asarray(trigger_ids, np.int64)
    other = np.setdiff1d(np.arange(vocab), trig)
    tok = other[(h % np.uint64(other.size)).astype(np.int64)]
    is_t = u < 1.0 / mean_span
    tok = np.where(is_t, trig[(h >> np.uint64(32)).astype(np.int64) % trig.size], tok)
    return tok.astype(np.int32)


def page_table(key, lengths_cap, page_size: int):
    """Seeded random page assignment. lengths_cap[b] = positions sequence b may reach.

    Returns (table [B][max_pages] int32 with -1 for unused, n_pages)."""
    need = [(int(c) + page_size - 1) // page_size for c in lengths_cap]
    n_pages = int(sum(need))
    hv = hash_at(key, STREAM_PAGE, 0, 0, 0, np.arange(n_pages), 0)
    perm = np.argsort(hv, kind="stable").astype(np.int32)
    max_pages = max(need)
    table = np.full((len(need), max_pages), -1, dtype=np.int32)
    o = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[o:o + n]
        o += n
    return table, n_pages
