// select.cu -- the SFI Selector (section 2B of the gist.science technical summary of
// "Slow-Fast Inference"): evidence f fused with a positional prior in the closed form
// s = (1 - lambda) f + lambda r, then Top-K positions, ties to the lower position.
//
// One CTA of 1024 threads per unit. The K-th largest score is found by an exact radix
// select on the scores' order-preserving 32-bit keys: a 12-bit digit over every candidate,
// then two 10-bit digits over the candidates gathered from the threshold's 12-bit bin
// (shared-memory histograms); one ordered pass then writes the chosen positions in
// ascending order with a single block-wide scan per chunk. The fused score uses
// round-to-nearest multiplies and adds with no contraction, so it is bit-reproducible on
// any IEEE host.
//
// When the unit's candidates fit (up to kStageCap evidence values), the evidence is first
// copied into shared memory (16-byte loads from every thread, all in flight together),
// turned into keys in place by the first pass, and every later pass reads the keys there;
// otherwise the passes stream it from global memory (L2-resident after the first) with
// eight loads per thread in flight.
#include <mutex>

#include "sfi_device.cuh"

namespace sfi {
namespace {

constexpr int NT = kSelectThreads;
constexpr int kWarps = NT / 32;
constexpr int kListCap = 8192;    // keys gathered for the refining passes
constexpr int kBatch = 8;         // candidates per thread per streaming step

__device__ __forceinline__ uint32_t order_key(float x)
{
    if (x != x)
        return 0u;
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Fused score key of candidate i (position n_sink + i) from its evidence value.
struct Fuse {
    int n;           // candidates
    float c1, c2, inv_tau;
    __device__ __forceinline__ uint32_t key(float fv, int i) const
    {
        const float rt = fminf(1.f, __fmul_rn(static_cast<float>(n - i), inv_tau));
        const float s = __fadd_rn(__fmul_rn(c1, fv), __fmul_rn(c2, rt));
        return order_key(s);
    }
};

// Constants of the fused score for nC candidates (the prior's closed-form normaliser Z in
// fp64, then rounded once): c[0] = fl32(1 - lambda), c[1] = fl32(lambda / Z),
// c[2] = fl32(1 / tau).
__device__ __forceinline__ void prior_consts(int nC, int tau, double lambda, float *c)
{
    const double Z = (nC >= tau) ? (tau + 1) * 0.5 + static_cast<double>(nC - tau)
                                 : static_cast<double>(nC) * (nC + 1) / (2.0 * tau);
    c[0] = __double2float_rn(1.0 - lambda);
    c[1] = __double2float_rn(lambda / Z);
    c[2] = __double2float_rn(1.0 / tau);
}

// Block-wide exclusive scan of one int per thread; returns the exclusive prefix and
// writes the block total to *total. Uses `scratch` (>= kWarps + 1 ints).
__device__ __forceinline__ int block_exclusive_scan(int x, int *scratch, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    if (lane == 31)
        scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kWarps ? scratch[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o)
                wi += y;
        }
        if (lane < kWarps)
            scratch[lane] = wi - w;
        if (lane == kWarps - 1)
            scratch[kWarps] = wi;
    }
    __syncthreads();
    const int r = scratch[warp] + incl - x;
    *total = scratch[kWarps];
    __syncthreads();
    return r;
}

// Dynamic shared memory: nsub sub-histograms of 4096 bins (warps w with w % nsub equal
// share one, so fewer lanes collide on a bin), the gathered list, then (staged mode) the
// evidence of the unit's candidates.
size_t select_smem_bytes(bool staged)
{
    return (static_cast<size_t>(staged ? 2 : 4) * 4096 + kListCap) * sizeof(uint32_t) +
           (staged ? static_cast<size_t>(kStageCap) * sizeof(float) : 0);
}

// Exclusive scan over the warps of the block of one (a, b) pair per warp, given by lane 0;
// returns the pair of the warps before this one (in every lane) and writes the totals.
// Uses `scratch` (>= 2 kWarps + 2 ints).
__device__ __forceinline__ int2 warp_totals_exclusive_scan(int a, int b, int *scratch, int2 *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        scratch[warp] = a;
        scratch[kWarps + warp] = b;
    }
    __syncthreads();
    if (warp == 0) {
        const int x = lane < kWarps ? scratch[lane] : 0;
        const int y = lane < kWarps ? scratch[kWarps + lane] : 0;
        int xi = x, yi = y;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int xu = __shfl_up_sync(0xffffffffu, xi, o);
            const int yu = __shfl_up_sync(0xffffffffu, yi, o);
            if (lane >= o) {
                xi += xu;
                yi += yu;
            }
        }
        __syncwarp();
        if (lane < kWarps) {
            scratch[lane] = xi - x;
            scratch[kWarps + lane] = yi - y;
        }
        if (lane == kWarps - 1) {
            scratch[2 * kWarps] = xi;
            scratch[2 * kWarps + 1] = yi;
        }
    }
    __syncthreads();
    const int2 r = make_int2(scratch[warp], scratch[kWarps + warp]);
    *total = make_int2(scratch[2 * kWarps], scratch[2 * kWarps + 1]);
    __syncthreads();
    return r;
}

// Digit of the histogram hist (nb = 4 NT or NT bins) where the running count from the top
// first reaches krem: the bin in *digit and the count above it in *above (shared memory).
// Thread t sums its nb / NT consecutive bins from the top (one 16-byte load for 4 NT bins);
// every warp then scans the 32 warp sums itself, so the search takes two barriers, the last
// of which publishes the result. Uses scratch[0, kWarps).
__device__ __forceinline__ void find_top_digit(const uint32_t *hist, int nb, int krem, int *scratch,
                                               uint32_t *digit, int *above)
{
    static_assert(kWarps == 32, "one warp sum per lane");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t hb[4] = {0u, 0u, 0u, 0u};   // this thread's bins, descending
    if (nb == 4 * NT) {
        const uint4 v = reinterpret_cast<const uint4 *>(hist)[NT - 1 - tid];
        hb[0] = v.w;
        hb[1] = v.z;
        hb[2] = v.y;
        hb[3] = v.x;
    } else {
        hb[0] = hist[NT - 1 - tid];
    }
    const int per = nb / NT;
    const int mine = static_cast<int>(hb[0] + hb[1] + hb[2] + hb[3]);
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    if (lane == 31)
        scratch[warp] = incl;
    __syncthreads();
    const int ws = scratch[lane];
    int wincl = ws;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wincl, o);
        if (lane >= o)
            wincl += y;
    }
    int before = __shfl_sync(0xffffffffu, wincl - ws, warp) + incl - mine;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int h = static_cast<int>(hb[j]);
        if (j < per && before < krem && before + h >= krem) {
            *digit = static_cast<uint32_t>(nb - 1 - (per * tid + j));
            *above = before;
        }
        before += h;
    }
    __syncthreads();
}

// Block-wide sum of one int per thread, in one barrier. Uses scratch[0, kWarps); the caller
// keeps the region untouched until every thread has returned.
__device__ __forceinline__ int block_total(int x, int *scratch)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0)
        scratch[warp] = x;
    __syncthreads();
    int t = scratch[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
}

// warp_totals_exclusive_scan in one barrier: every warp scans the 32 pairs itself. Uses
// scratch[0, 2 kWarps); the caller keeps the region untouched until every thread has returned.
__device__ __forceinline__ int2 warp_pairs_exclusive_scan(int a, int b, int *scratch, int2 *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        scratch[warp] = a;
        scratch[kWarps + warp] = b;
    }
    __syncthreads();
    const int x = scratch[lane], y = scratch[kWarps + lane];
    int xi = x, yi = y;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int xu = __shfl_up_sync(0xffffffffu, xi, o);
        const int yu = __shfl_up_sync(0xffffffffu, yi, o);
        if (lane >= o) {
            xi += xu;
            yi += yu;
        }
    }
    *total = make_int2(__shfl_sync(0xffffffffu, xi, 31), __shfl_sync(0xffffffffu, yi, 31));
    return make_int2(__shfl_sync(0xffffffffu, xi - x, warp), __shfl_sync(0xffffffffu, yi - y, warp));
}

// At most 56 registers per thread: a 1024-thread CTA then takes 7/8 of the register file
// instead of all of it, so a launch under a profiler, which may need a few more, still fits.
__global__ void __maxnreg__(56) select_kernel(const SelectParams p)
{
    __shared__ int scratch[2 * kWarps + 2];
    __shared__ uint32_t sh_digit;
    __shared__ int sh_above;
    __shared__ int sh_count;
    __shared__ float sh_c[3];

    // Dependents start only once the selection is written (pdl_trigger_after_writes): the
    // fast step reads the packed memory that follows from it before its own wait.
    const int tid = threadIdx.x, lane = tid & 31;
    pdl_wait();
    const int u = launched_unit(static_cast<int>(blockIdx.x), p.n_seq_active, p.active, p.batch,
                                p.n_kv_heads);
    if (u < 0)
        return;
    const int b = (u / p.n_kv_heads) % p.batch;
    if (p.active && !p.active[b])
        return;
    const int L0 = p.seq_len[b];
    if (L0 < 0 || L0 > p.max_len) {   // outside the caller's bound: no selection
        if (tid == 0)
            raise_error(p.err, 0x8u);  // SFI_DEVERR_LENGTH
        return;
    }
    const int L = min(L0, p.capacity);
    const int S = p.n_sink, W = p.n_window;
    const int nC = max(0, L - W - S);
    const int K = min(p.n_select, nC);
    int32_t *out = p.sel_idx + static_cast<size_t>(u) * p.n_select;
    if (K == nC) {  // every candidate is kept (includes K == 0)
        for (int i = tid; i < nC; i += NT)
            out[i] = S + i;
        if (tid == 0)
            p.sel_cnt[u] = nC;
        __syncthreads();
        pdl_trigger_after_writes();
        return;
    }
    const float *fg = p.f + static_cast<size_t>(u) * p.capacity + S;
    Fuse fz;
    fz.n = nC;
    // fp64 is slow here: one thread computes the prior's constants, published by the
    // barrier that ends the staging
    if (tid == 0)
        prior_consts(nC, p.prior_tau, p.lambda, sh_c);

    extern __shared__ __align__(16) uint32_t dyn[];
    const int nsub = p.staged ? 2 : 4;
    uint32_t *hist = dyn;
    uint32_t *lst = dyn + nsub * 4096;
    float *fs = reinterpret_cast<float *>(lst + kListCap);
    const int sub = (tid >> 5) % nsub;

    // ---- staged mode: the candidates' evidence into shared memory -----------------------
    // The copy starts at the 16-byte boundary at or below the first candidate (f is 16-byte
    // aligned, so this stays inside the buffer) and ends at most 12 bytes past the last one
    // (the host stages only when that stays inside the unit's row).
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(fg);
    const int off = p.staged ? static_cast<int>((a0 & 15u) >> 2) : 0;
    const bool staged = p.staged && off + nC <= kStageCap;
    if (staged) {
        // every thread copies its 16-byte pieces; all loads are in flight before any store
        const uint4 *src = reinterpret_cast<const uint4 *>(fg - off);
        uint4 *dst = reinterpret_cast<uint4 *>(fs);
        const int n16 = ((off + nC) * 4 + 15) >> 4;
        for (int b0 = 0; b0 < n16; b0 += 8 * NT) {
            uint4 x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int i = b0 + e * NT + tid;
                if (i < n16)
                    x[e] = src[i];
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int i = b0 + e * NT + tid;
                if (i < n16)
                    dst[i] = x[e];
            }
        }
    }
    for (int i = tid; i < nsub * 4096; i += NT)
        hist[i] = 0u;
    if (tid == 0)
        sh_count = 0;
    __syncthreads();
    fz.c1 = sh_c[0];
    fz.c2 = sh_c[1];
    fz.inv_tau = sh_c[2];

    // staged mode: pass 0 turns each staged evidence value into its key in place, and the
    // later passes read the keys; streaming mode recomputes keys from global memory
    uint32_t *ks = reinterpret_cast<uint32_t *>(fs) + off;
    bool keys_ready = false;
    auto key_at = [&](int i) -> uint32_t {
        return keys_ready ? ks[i] : fz.key(staged ? fs[off + i] : __ldg(fg + i), i);
    };
    int nbins = 4096;
    auto count = [&](bool part, uint32_t digit) {
        if (part)
            atomicAdd(&hist[sub * nbins + digit], 1u);
    };
    // the bin, scanning from the top, where the running count first reaches krem
    auto bin_count = [&](int bin) {
        int h = 0;
        for (int s2 = 0; s2 < nsub; ++s2)
            h += static_cast<int>(hist[s2 * nbins + bin]);
        return h;
    };
    auto find_digit = [&](int nb, int krem_now) {
        const int per = nb / NT;
        int mine = 0;
        for (int j = 0; j < per; ++j)
            mine += bin_count(nb - 1 - (per * tid + j));
        int total;
        int before = block_exclusive_scan(mine, scratch, &total);
        for (int j = 0; j < per; ++j) {
            const int bin = nb - 1 - (per * tid + j);
            const int h = bin_count(bin);
            if (before < krem_now && before + h >= krem_now) {
                sh_digit = static_cast<uint32_t>(bin);
                sh_above = before;
            }
            before += h;
        }
        __syncthreads();
    };
    // keys of candidates base + e * NT + tid, e < kBatch (all loads in flight together)
    auto load_batch = [&](int base, uint32_t (&k)[kBatch]) {
        if (keys_ready) {
#pragma unroll
            for (int e = 0; e < kBatch; ++e) {
                const int i = base + e * NT + tid;
                k[e] = i < nC ? ks[i] : 0u;
            }
            return;
        }
        float v[kBatch];
#pragma unroll
        for (int e = 0; e < kBatch; ++e) {
            const int i = base + e * NT + tid;
            v[e] = i < nC ? (staged ? fs[off + i] : __ldg(fg + i)) : 0.f;
        }
#pragma unroll
        for (int e = 0; e < kBatch; ++e)
            k[e] = fz.key(v[e], base + e * NT + tid);
    };

    // ---- radix select of the K-th largest key ------------------------------------------
    // pass 0: top 12 bits of every candidate
    for (int base = 0; base < nC; base += kBatch * NT) {
        uint32_t k[kBatch];
        load_batch(base, k);
#pragma unroll
        for (int e = 0; e < kBatch; ++e) {
            const int i = base + e * NT + tid;
            if (staged && i < nC)
                ks[i] = k[e];  // each thread overwrites only values it has read itself
            count(i < nC, k[e] >> 20);
        }
    }
    __syncthreads();
    keys_ready = staged;
    int krem = K;
    find_digit(4096, krem);
    const uint32_t d0 = sh_digit;
    uint32_t prefix = d0 << 20, pmask = 0xFFF00000u;
    krem -= sh_above;
    const int n_lst = bin_count(static_cast<int>(d0));
    const bool use_list = n_lst <= kListCap;
    __syncthreads();
    if (use_list) {
        for (int base = 0; base < nC; base += kBatch * NT) {
            uint32_t k[kBatch];
            load_batch(base, k);
#pragma unroll
            for (int e = 0; e < kBatch; ++e) {
                const bool in = base + e * NT + tid < nC && (k[e] >> 20) == d0;
                const unsigned bal = __ballot_sync(0xffffffffu, in);
                int wbase = 0;
                if (lane == 0 && bal)
                    wbase = atomicAdd(&sh_count, __popc(bal));
                wbase = __shfl_sync(0xffffffffu, wbase, 0);
                if (in)
                    lst[wbase + __popc(bal & ((1u << lane) - 1u))] = k[e];
            }
        }
        __syncthreads();
    }
    // passes 1 and 2: 10-bit digits, over the gathered list (or every candidate)
#pragma unroll 1
    for (int pass = 1; pass < 3; ++pass) {
        const int shift = pass == 1 ? 10 : 0;
        nbins = 1024;
        for (int i = tid; i < nsub * 1024; i += NT)
            hist[i] = 0u;
        __syncthreads();
        if (use_list) {
            for (int base = 0; base < n_lst; base += NT) {
                const int i = base + tid;
                const uint32_t k = i < n_lst ? lst[i] : 0u;
                count(i < n_lst && (k & pmask) == prefix, (k >> shift) & 1023u);
            }
        } else {
            for (int base = 0; base < nC; base += kBatch * NT) {
                uint32_t k[kBatch];
                load_batch(base, k);
#pragma unroll
                for (int e = 0; e < kBatch; ++e)
                    count(base + e * NT + tid < nC && (k[e] & pmask) == prefix,
                          (k[e] >> shift) & 1023u);
            }
        }
        __syncthreads();
        find_digit(1024, krem);
        prefix |= sh_digit << shift;
        pmask |= 1023u << shift;
        krem -= sh_above;
        __syncthreads();
    }
    const uint32_t thr = prefix;  // exact key of the K-th largest score
    const int need_eq = krem;     // how many keys equal to thr are taken (lowest first)

    // ---- ordered compaction ------------------------------------------------------------
    // A chosen candidate's slot = (keys > thr before it) + min(keys == thr before it,
    // need_eq). Warp w takes one contiguous range of candidates, 32 per step (lane =
    // candidate): ballots count its greater and equal keys; one scan over the warps gives
    // every warp its starting counts; a second pass over its keys writes the chosen
    // positions in ascending order.
    {
        const int warp = tid >> 5;
        const unsigned lt_mask = (1u << lane) - 1u;
        const int span = (nC + kWarps * 32 - 1) / (kWarps * 32) * 32;  // per warp
        const int w0 = warp * span, w1 = min(nC, w0 + span);
        int n_gt = 0, n_eq = 0;
        for (int i0 = w0; i0 < w1; i0 += 32) {
            const int i = i0 + lane;
            const bool in = i < w1;
            const uint32_t k = in ? key_at(i) : 0u;
            n_gt += __popc(__ballot_sync(0xffffffffu, in && k > thr));
            n_eq += __popc(__ballot_sync(0xffffffffu, in && k == thr));
        }
        int2 tot;
        const int2 before = warp_totals_exclusive_scan(n_gt, n_eq, scratch, &tot);
        int gt_before = before.x, eq_before = before.y;
        for (int i0 = w0; i0 < w1; i0 += 32) {
            const int i = i0 + lane;
            const bool in = i < w1;
            const uint32_t k = in ? key_at(i) : 0u;
            const unsigned gm = __ballot_sync(0xffffffffu, in && k > thr);
            const unsigned em = __ballot_sync(0xffffffffu, in && k == thr);
            const int g_lt = gt_before + __popc(gm & lt_mask);
            const int e_lt = eq_before + __popc(em & lt_mask);
            if ((gm >> lane) & 1u)
                out[g_lt + min(e_lt, need_eq)] = S + i;
            else if (((em >> lane) & 1u) && e_lt < need_eq)
                out[g_lt + e_lt] = S + i;
            gt_before += __popc(gm);
            eq_before += __popc(em);
        }
    }
    if (tid == 0) {
        p.sel_cnt[u] = K;
    }
    __syncthreads();
    pdl_trigger_after_writes();
}

// ---------------------------------------------------------------------------------------
// Clustered Selector: the C CTAs of a cluster share one unit. CTA r stages the evidence of
// candidates [r nC / C, (r+1) nC / C) in its shared memory, turns it into keys, and builds
// a local histogram per radix pass; after one cluster barrier every CTA sums all C local
// histograms through distributed shared memory and finds the same digit. Histograms are
// double-buffered, so a CTA that has passed pass p's barrier never overwrites a buffer a peer
// may still read. The ordered output exchanges each CTA's (greater, equal) counts the same
// way. Every CTA of a cluster runs every barrier: the only early exits (inactive sequence,
// all candidates kept) are taken by all of them together.

constexpr int kClusterKeyCap = 33280;  // candidates per CTA (a 131K context in 4 CTAs)
static_assert(kClusterKeyCap < 65536, "a CTA's first-pass counts are packed in 16 bits");
constexpr int kMergeCap = 4096;        // threshold-bin keys exchanged as lists (else radix)
constexpr int kMaxCluster = 4;         // CTAs per unit (the host picks 4 or 2)
static_assert(NT == 1024, "the cluster's histogram passes take 4096 and 1024 bins");

size_t select_cluster_smem_bytes()
{
    // keys: up to kClusterKeyCap candidates, 3 words of alignment slack before them and up
    // to 3 after (the copy is whole 16-byte pieces)
    return (3 * 4096 + 2048 + kClusterKeyCap + 8) * sizeof(uint32_t);
}

__global__ void __maxnreg__(56) select_cluster_kernel(const SelectParams p)
{
    __shared__ int scratch[2 * kWarps + 2];    // digit searches and the compaction's scan
    __shared__ int scratch2[2 * kWarps];       // the list path's totals and scan
    __shared__ uint32_t sh_digit;
    __shared__ int sh_above;
    __shared__ int sh_counts[2];  // this CTA's (greater, equal) keys for the ordered output,
                                  // or (keys above the threshold bin, its list length)
    __shared__ int sh_lcnt;
    __shared__ float sh_c[3];

    // dependents start only once the selection is written (see select_kernel)
    pdl_wait();
    const int C = p.cluster;
    const int rank = static_cast<int>(blockIdx.x) % C;
    const int u = launched_unit(static_cast<int>(blockIdx.x) / C, p.n_seq_active, p.active,
                                p.batch, p.n_kv_heads);
    if (u < 0)
        return;   // (every CTA of the cluster alike: no cluster barrier is reached)
    const int b = (u / p.n_kv_heads) % p.batch;
    if (p.active && !p.active[b])
        return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L0 = p.seq_len[b];
    // outside the caller's bound (which sized the shared-memory staging): no selection, in
    // every CTA of the cluster alike
    if (L0 < 0 || L0 > p.max_len) {
        if (tid == 0 && rank == 0)
            raise_error(p.err, 0x8u);  // SFI_DEVERR_LENGTH
        return;
    }
    const int L = min(L0, p.capacity);
    const int S = p.n_sink, W = p.n_window;
    const int nC = max(0, L - W - S);
    const int K = min(p.n_select, nC);
    const int c0 = static_cast<int>(static_cast<long long>(rank) * nC / C);
    const int c1 = static_cast<int>(static_cast<long long>(rank + 1) * nC / C);
    const int nloc = c1 - c0;
    int32_t *out = p.sel_idx + static_cast<size_t>(u) * p.n_select;
    if (K == nC) {  // every candidate is kept (includes K == 0)
        for (int i = c0 + tid; i < c1; i += NT)
            out[i] = S + i;
        if (tid == 0 && rank == 0)
            p.sel_cnt[u] = nC;
        __syncthreads();
        pdl_trigger_after_writes();
        return;
    }
    Fuse fz;
    fz.n = nC;
    // fp64 is slow here: one thread computes the prior's constants, published by the
    // barrier that ends the staging
    if (tid == 0)
        prior_consts(nC, p.prior_tau, p.lambda, sh_c);

    extern __shared__ __align__(16) uint32_t dyn[];
    uint32_t *hbuf0 = dyn, *hbuf1 = dyn + 4096;  // local histograms, by pass parity
    uint32_t *gsum = dyn + 2 * 4096;             // the cluster's sums
    uint32_t *hpk = dyn + 3 * 4096;              // the first pass's counts, packed for the peers
    uint32_t *kraw = dyn + 3 * 4096 + 2048;      // staged evidence, then keys

    // ---- stage this CTA's candidates (16-byte loads, all in flight together) ------------
    // With p.zbuf (group of 4) the evidence is computed here from the dense step's logits
    // (one 16-byte load of four heads per candidate, the first 4 NT requested now) and the
    // merged statistics, term for term as the evidence pass computes it, and written to
    // p.f_out; otherwise the evidence pass's output is copied in.
    const bool fev = p.zbuf != nullptr;
    __shared__ float sh_M[4], sh_inv[4];
    float4 zr[4];
    const float *fg = p.f + static_cast<size_t>(u) * p.capacity + S + c0;
    const int off = fev ? 0 : static_cast<int>((reinterpret_cast<uintptr_t>(fg) & 15u) >> 2);
    const float4 *zg = fev ? reinterpret_cast<const float4 *>(p.zbuf) +
                                 (static_cast<size_t>(u) * p.capacity + S + c0)
                           : nullptr;
    if (fev) {
        if (tid < 4) {
            const float2 st = __ldcg(p.stats + static_cast<size_t>(u) * 4 + tid);
            sh_M[tid] = st.x;
            sh_inv[tid] = st.y > 0.f ? 1.f / st.y : 0.f;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = e * NT + tid;
            if (i < nloc)
                zr[e] = __ldcg(zg + i);
        }
    } else {
        const uint4 *src = reinterpret_cast<const uint4 *>(fg - off);
        uint4 *dst = reinterpret_cast<uint4 *>(kraw);
        const int n16 = ((off + nloc) * 4 + 15) >> 4;
        for (int b0 = 0; b0 < n16; b0 += 4 * NT) {
            uint4 x[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = b0 + e * NT + tid;
                if (i < n16)
                    x[e] = src[i];
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = b0 + e * NT + tid;
                if (i < n16)
                    dst[i] = x[e];
            }
        }
    }
    for (int i = tid; i < 4096; i += NT)
        hbuf0[i] = 0u;
    __syncthreads();
    fz.c1 = sh_c[0];
    fz.c2 = sh_c[1];
    fz.inv_tau = sh_c[2];
    uint32_t *ks = kraw + off;  // ks[i] = key of candidate c0 + i

    // ---- pass 0: keys in place, top-12-bit histogram --------------------------------------
    if (fev) {
        const float M0 = sh_M[0], M1 = sh_M[1], M2 = sh_M[2], M3 = sh_M[3];
        const float i0v = sh_inv[0], i1v = sh_inv[1], i2v = sh_inv[2], i3v = sh_inv[3];
        float *fo = p.f_out + static_cast<size_t>(u) * p.capacity + S + c0;
        for (int b0 = 0; b0 < nloc; b0 += 4 * NT) {
            if (b0 > 0) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = b0 + e * NT + tid;
                    if (i < nloc)
                        zr[e] = __ldcg(zg + i);
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = b0 + e * NT + tid;
                if (i < nloc) {
                    float acc = 0.f;
                    acc = fmaf(exp2f(zr[e].x - M0), i0v, acc);
                    acc = fmaf(exp2f(zr[e].y - M1), i1v, acc);
                    acc = fmaf(exp2f(zr[e].z - M2), i2v, acc);
                    acc = fmaf(exp2f(zr[e].w - M3), i3v, acc);
                    const float fv = acc * 0.25f;
                    fo[i] = fv;
                    const uint32_t k = fz.key(fv, c0 + i);
                    ks[i] = k;
                    atomicAdd(&hbuf0[k >> 20], 1u);
                }
            }
        }
    } else {
        for (int i = tid; i < nloc; i += NT) {
            const uint32_t k = fz.key(__uint_as_float(ks[i]), c0 + i);
            ks[i] = k;
            atomicAdd(&hbuf0[k >> 20], 1u);
        }
    }
    // the counts packed for the exchange in 16 bits, bins 2j and 2j + 1 in the low and high
    // half of word j (a CTA holds at most kClusterKeyCap < 2^16 keys): the peers then read
    // half the bytes (counting into packed words directly was slower: the few occupied bins
    // collide)
    __syncthreads();
    {
        const uint4 h4 = reinterpret_cast<const uint4 *>(hbuf0)[tid];
        reinterpret_cast<uint2 *>(hpk)[tid] = make_uint2((h4.x & 0xFFFFu) | (h4.y << 16),
                                                         (h4.z & 0xFFFFu) | (h4.w << 16));
    }
    // digit of the histogram hist (nb bins) where the running count from the top first
    // reaches krem (sh_digit, and the count above it in sh_above; two barriers)
    auto find_digit = [&](const uint32_t *hist, int nb, int krem_now) {
        find_top_digit(hist, nb, krem_now, scratch, &sh_digit, &sh_above);
    };
    // the same over the cluster's summed histogram; every CTA computes the same digit
    // (this thread's nb / NT bins, 4 consecutive ones for the 4096-bin pass, from each of the
    // C <= 4 CTAs: one 8-byte remote load of packed 16-bit counts per CTA for the 4096-bin
    // pass, all issued before the first is used; the sums in 32 bits)
    auto merged_digit = [&](const uint32_t *mine, int nb, int krem_now) {
        cluster_sync_all();  // every CTA's local histogram of this pass is complete
        if (nb == 4 * NT) {
            uint2 v[kMaxCluster];
#pragma unroll
            for (int r = 0; r < kMaxCluster; ++r)
                v[r] = r < C ? ld_cluster_v2_u32(map_to_rank(mine + 2 * tid, static_cast<uint32_t>(r)))
                             : make_uint2(0u, 0u);
            uint4 h = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int r = 0; r < kMaxCluster; ++r) {
                h.x += v[r].x & 0xFFFFu;
                h.y += v[r].x >> 16;
                h.z += v[r].y & 0xFFFFu;
                h.w += v[r].y >> 16;
            }
            reinterpret_cast<uint4 *>(gsum)[tid] = h;
        } else {
            uint32_t v[kMaxCluster];
#pragma unroll
            for (int r = 0; r < kMaxCluster; ++r)
                v[r] = r < C ? ld_cluster_u32(map_to_rank(mine + tid, static_cast<uint32_t>(r))) : 0u;
            uint32_t h = 0;
#pragma unroll
            for (int r = 0; r < kMaxCluster; ++r)
                h += v[r];
            gsum[tid] = h;
        }
        __syncthreads();
        find_digit(gsum, nb, krem_now);
    };
    int krem = K;
    merged_digit(hpk, 4096, krem);
    const uint32_t d0 = sh_digit;
    uint32_t prefix = d0 << 20, pmask = 0xFFF00000u;
    krem -= sh_above;
    const unsigned lt_mask = (1u << lane) - 1u;
    // The unit's keys in the threshold's 12-bit bin: usually few. Then every CTA gathers its
    // own into a list, the lists are exchanged once, and each CTA finishes the exact
    // threshold on the merged list alone (the same result in every CTA), and takes the
    // counts of the CTAs before it from the lists too. Otherwise (many ties) the remaining
    // two 10-bit digits are found over the cluster's summed histograms.
    const bool listed = static_cast<int>(gsum[d0]) <= kMergeCap;   // the same in every CTA
    int gt_before = 0, eq_before = 0;  // keys above / equal to the threshold in earlier CTAs
    if (listed) {
        if (tid == 0)
            sh_lcnt = 0;
        __syncthreads();
        int above = 0;  // this thread's keys above the threshold bin
        for (int i0 = 0; i0 < nloc; i0 += NT) {
            const int i = i0 + tid;
            const uint32_t k = i < nloc ? ks[i] : 0u;
            const bool in = i < nloc && (k >> 20) == d0;
            above += (i < nloc && (k >> 20) > d0) ? 1 : 0;
            const unsigned bal = __ballot_sync(0xffffffffu, in);
            int wbase = 0;
            if (lane == 0 && bal)
                wbase = atomicAdd(&sh_lcnt, __popc(bal));
            wbase = __shfl_sync(0xffffffffu, wbase, 0);
            if (in)
                hbuf1[wbase + __popc(bal & lt_mask)] = k;
        }
        const int tot_above = block_total(above, scratch2);
        if (tid == 0) {
            sh_counts[0] = tot_above;
            sh_counts[1] = sh_lcnt;
        }
        cluster_sync_all();  // every CTA's list and counts are in place
        // the merged list in hbuf0 (free now: the peers read the packed copy), the
        // CTAs' lists in rank order; the lists before this CTA's end at `mine0`
        int lens[kMaxCluster], gts[kMaxCluster];
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) {
            lens[r] = r < C ? static_cast<int>(ld_cluster_u32(map_to_rank(&sh_counts[1], static_cast<uint32_t>(r)))) : 0;
            gts[r] = r < C ? static_cast<int>(ld_cluster_u32(map_to_rank(&sh_counts[0], static_cast<uint32_t>(r)))) : 0;
        }
        int n_all = 0, mine0 = 0, longest = 0, starts[kMaxCluster];
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) {
            starts[r] = n_all;
            if (r < rank)
                gt_before += gts[r];
            if (r == rank)
                mine0 = n_all;
            n_all += lens[r];
            longest = max(longest, lens[r]);
        }
        for (int i = tid; i < longest; i += NT) {
            uint32_t x[kMaxCluster];
#pragma unroll
            for (int r = 0; r < kMaxCluster; ++r)
                x[r] = i < lens[r] ? ld_cluster_u32(map_to_rank(hbuf1 + i, static_cast<uint32_t>(r))) : 0u;
#pragma unroll
            for (int r = 0; r < kMaxCluster; ++r)
                if (i < lens[r])
                    hbuf0[starts[r] + i] = x[r];
        }
        // passes 1 and 2 (10-bit digits) over the merged list: 1024-bin histograms in
        // gsum[0, 1024) and gsum[1024, 2048), zeroed together (the digit search's last barrier
        // publishes each digit before the next pass reads it)
        gsum[tid] = 0u;
        gsum[NT + tid] = 0u;
        __syncthreads();
#pragma unroll 1
        for (int pass = 1; pass < 3; ++pass) {
            const int shift = pass == 1 ? 10 : 0;
            uint32_t *hp = gsum + (pass - 1) * NT;
            for (int i = tid; i < n_all; i += NT) {
                const uint32_t k = hbuf0[i];
                if ((k & pmask) == prefix)
                    atomicAdd(&hp[(k >> shift) & 1023u], 1u);
            }
            __syncthreads();
            find_digit(hp, 1024, krem);
            prefix |= sh_digit << shift;
            pmask |= 1023u << shift;
            krem -= sh_above;
        }
        // keys above and equal to the threshold in the lists of the CTAs before this one
        int cg = 0, ce = 0;
        for (int i = tid; i < mine0; i += NT) {
            const uint32_t k = hbuf0[i];
            cg += k > prefix ? 1 : 0;
            ce += k == prefix ? 1 : 0;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            cg += __shfl_xor_sync(0xffffffffu, cg, o);
            ce += __shfl_xor_sync(0xffffffffu, ce, o);
        }
        int2 tot2;
        warp_pairs_exclusive_scan(cg, ce, scratch2, &tot2);
        gt_before += tot2.x;
        eq_before += tot2.y;
    } else {
        // passes 1 and 2: 10-bit digits over this CTA's keys that share the prefix
#pragma unroll 1
        for (int pass = 1; pass < 3; ++pass) {
            const int shift = pass == 1 ? 10 : 0;
            uint32_t *hb = (pass & 1) ? hbuf1 : hbuf0;
            for (int i = tid; i < 1024; i += NT)
                hb[i] = 0u;
            __syncthreads();
            for (int i = tid; i < nloc; i += NT) {
                const uint32_t k = ks[i];
                if ((k & pmask) == prefix)
                    atomicAdd(&hb[(k >> shift) & 1023u], 1u);
            }
            merged_digit(hb, 1024, krem);
            prefix |= sh_digit << shift;
            pmask |= 1023u << shift;
            krem -= sh_above;
            __syncthreads();
        }
    }
    const uint32_t thr = prefix;  // exact key of the K-th largest score
    const int need_eq = krem;     // how many keys equal to thr are taken (lowest first)

    // ---- ordered compaction (as in select_kernel, offset by the CTAs before this one) ----
    const int span = (nloc + kWarps * 32 - 1) / (kWarps * 32) * 32;
    const int w0 = warp * span, w1 = min(nloc, w0 + span);
    int n_gt = 0, n_eq = 0;
    for (int i0 = w0; i0 < w1; i0 += 32) {
        const int i = i0 + lane;
        const bool in = i < w1;
        const uint32_t k = in ? ks[i] : 0u;
        n_gt += __popc(__ballot_sync(0xffffffffu, in && k > thr));
        n_eq += __popc(__ballot_sync(0xffffffffu, in && k == thr));
    }
    int2 tot;
    const int2 before = warp_pairs_exclusive_scan(n_gt, n_eq, scratch, &tot);
    if (!listed) {
        if (tid == 0) {
            sh_counts[0] = tot.x;
            sh_counts[1] = tot.y;
        }
        cluster_sync_all();  // every CTA's counts are in place
        uint32_t g4[kMaxCluster], e4[kMaxCluster];
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) {
            g4[r] = r < rank ? ld_cluster_u32(map_to_rank(&sh_counts[0], static_cast<uint32_t>(r))) : 0u;
            e4[r] = r < rank ? ld_cluster_u32(map_to_rank(&sh_counts[1], static_cast<uint32_t>(r))) : 0u;
        }
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) {
            gt_before += static_cast<int>(g4[r]);
            eq_before += static_cast<int>(e4[r]);
        }
    }
    gt_before += before.x;
    eq_before += before.y;
    for (int i0 = w0; i0 < w1; i0 += 32) {
        const int i = i0 + lane;
        const bool in = i < w1;
        const uint32_t k = in ? ks[i] : 0u;
        const unsigned gm = __ballot_sync(0xffffffffu, in && k > thr);
        const unsigned em = __ballot_sync(0xffffffffu, in && k == thr);
        const int g_lt = gt_before + __popc(gm & lt_mask);
        const int e_lt = eq_before + __popc(em & lt_mask);
        if ((gm >> lane) & 1u)
            out[g_lt + min(e_lt, need_eq)] = S + c0 + i;
        else if (((em >> lane) & 1u) && e_lt < need_eq)
            out[g_lt + e_lt] = S + c0 + i;
        gt_before += __popc(gm);
        eq_before += __popc(em);
    }
    if (tid == 0 && rank == 0)
        p.sel_cnt[u] = K;
    __syncthreads();
    pdl_trigger_after_writes();
    cluster_sync_all();  // no CTA leaves while a peer may still read its shared memory
}

template <typename Kern>
int max_select_clusters(Kern kern, int cluster, size_t smem)
{
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cluster) * 64u);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

std::mutex g_sel_mu;
int g_sel_fit[64][9];  // max active clusters + 1 (0 = not yet queried)

}  // namespace

int select_cluster_size(int max_cluster)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 1;
    for (int C = 4; C >= 2; C >>= 1) {
        if (C > max_cluster)
            continue;
        int n;
        {
            std::lock_guard<std::mutex> lock(g_sel_mu);
            n = g_sel_fit[dev][C] - 1;
        }
        if (n < 0) {
            n = max_select_clusters(select_cluster_kernel, C, select_cluster_smem_bytes());
            std::lock_guard<std::mutex> lock(g_sel_mu);
            g_sel_fit[dev][C] = n + 1;
        }
        if (n >= 1)
            return C;
    }
    return 1;
}

int select_cluster_key_cap() { return kClusterKeyCap; }

cudaError_t launch_select(const SelectParams &p, cudaStream_t stream)
{
    if (p.cluster > 1) {
        const size_t smem = select_cluster_smem_bytes();
        const cudaError_t a = cudaFuncSetAttribute(select_cluster_kernel,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (a != cudaSuccess)
            return a;
        const cudaError_t e = launch_pdl_cluster(select_cluster_kernel, dim3(p.n_units * p.cluster),
                                                 dim3(NT), smem, p.cluster, stream, p);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    const size_t smem = select_smem_bytes(p.staged != 0);
    {
        const cudaError_t a =
            cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (a != cudaSuccess)
            return a;
    }
    const cudaError_t e = launch_pdl(select_kernel, dim3(p.n_units), dim3(NT), smem, stream, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace sfi
