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
// copied into shared memory with bulk asynchronous copies and every pass reads it there;
// otherwise the passes stream it from global memory (L2-resident after the first) with
// eight loads per thread in flight.
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

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar` (transaction
// bytes). Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Dynamic shared memory: nsub sub-histograms of 4096 bins (warps w with w % nsub equal
// share one, so fewer lanes collide on a bin), the gathered list, then (staged mode) the
// evidence of the unit's candidates.
size_t select_smem_bytes(bool staged)
{
    return (static_cast<size_t>(staged ? 2 : 4) * 4096 + kListCap) * sizeof(uint32_t) +
           (staged ? static_cast<size_t>(kStageCap) * sizeof(float) : 0);
}

// At most 56 registers per thread: a 1024-thread CTA then takes 7/8 of the register file
// instead of all of it, so a launch under a profiler, which may need a few more, still fits.
__global__ void __maxnreg__(56) select_kernel(const SelectParams p)
{
    __shared__ int scratch[kWarps + 1];
    __shared__ uint32_t sh_digit;
    __shared__ int sh_above;
    __shared__ int sh_count;
    __shared__ __align__(8) uint64_t stage_bar;

    pdl_trigger();
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid == 0) {
        mbar_init(&stage_bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    pdl_wait();
    const int u = blockIdx.x;
    const int b = (u / p.n_kv_heads) % p.batch;
    if (p.active && !p.active[b])
        return;
    const int L = min(p.seq_len[b], p.capacity);
    const int S = p.n_sink, W = p.n_window;
    const int nC = max(0, L - W - S);
    const int K = min(p.n_select, nC);
    int32_t *out = p.sel_idx + static_cast<size_t>(u) * p.n_select;
    if (K == nC) {  // every candidate is kept (includes K == 0)
        for (int i = tid; i < nC; i += NT)
            out[i] = S + i;
        if (tid == 0)
            p.sel_cnt[u] = nC;
        return;
    }
    const float *fg = p.f + static_cast<size_t>(u) * p.capacity + S;
    Fuse fz;
    fz.n = nC;
    const int tau = p.prior_tau;
    const double Z = (nC >= tau) ? (tau + 1) * 0.5 + static_cast<double>(nC - tau)
                                 : static_cast<double>(nC) * (nC + 1) / (2.0 * tau);
    fz.c1 = __double2float_rn(1.0 - p.lambda);
    fz.c2 = __double2float_rn(p.lambda / Z);
    fz.inv_tau = __double2float_rn(1.0 / tau);

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
    if (staged && tid == 0) {
        const char *src = reinterpret_cast<const char *>(fg - off);
        const uint32_t bytes = static_cast<uint32_t>(((off + nC) * 4 + 15) & ~15);
        mbar_arrive_expect_tx(&stage_bar, bytes);
        constexpr uint32_t kChunk = 16384;
        for (uint32_t o = 0; o < bytes; o += kChunk)
            bulk_load(reinterpret_cast<char *>(fs) + o, src + o,
                      bytes - o < kChunk ? bytes - o : kChunk, &stage_bar);
    }
    for (int i = tid; i < nsub * 4096; i += NT)
        hist[i] = 0u;
    if (tid == 0)
        sh_count = 0;
    if (staged && !mbar_wait(&stage_bar, 0, nullptr)) {
        // gave up: report, let the copies land (bounded again) and leave
        raise_error(p.err, 0x4u);  // SFI_DEVERR_TIMEOUT
        mbar_wait(&stage_bar, 0, nullptr);
        return;
    }
    __syncthreads();

    auto fval = [&](int i) -> float { return staged ? fs[off + i] : __ldg(fg + i); };
    auto key_at = [&](int i) -> uint32_t { return fz.key(fval(i), i); };
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
        float v[kBatch];
#pragma unroll
        for (int e = 0; e < kBatch; ++e) {
            const int i = base + e * NT + tid;
            v[e] = i < nC ? fval(i) : 0.f;
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
        for (int e = 0; e < kBatch; ++e)
            count(base + e * NT + tid < nC, k[e] >> 20);
    }
    __syncthreads();
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
    // need_eq), so one block scan of packed (equal << 16 | greater) counts per chunk of
    // 8 x NT candidates places every chosen index in ascending order.
    int gt_base = 0, eq_base = 0;
    for (int base = 0; base < nC; base += 8 * NT) {
        uint32_t k[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int i = base + 8 * tid + e;
            k[e] = i < nC ? key_at(i) : 0u;
        }
        int n_gt = 0, n_eq = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const bool in = base + 8 * tid + e < nC;
            n_gt += (in && k[e] > thr) ? 1 : 0;
            n_eq += (in && k[e] == thr) ? 1 : 0;
        }
        int tot;
        const int packed = block_exclusive_scan((n_eq << 16) | n_gt, scratch, &tot);
        int gt_before = gt_base + (packed & 0xFFFF);
        int eq_before = eq_base + (packed >> 16);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int i = base + 8 * tid + e;
            if (i >= nC)
                break;
            if (k[e] > thr) {
                out[gt_before + min(eq_before, need_eq)] = S + i;
                ++gt_before;
            } else if (k[e] == thr) {
                if (eq_before < need_eq)
                    out[gt_before + eq_before] = S + i;
                ++eq_before;
            }
        }
        gt_base += tot & 0xFFFF;
        eq_base += tot >> 16;
    }
    if (tid == 0)
        p.sel_cnt[u] = K;
}

}  // namespace

cudaError_t launch_select(const SelectParams &p, cudaStream_t stream)
{
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
