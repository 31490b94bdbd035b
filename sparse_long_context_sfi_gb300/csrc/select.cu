// select.cu -- the SFI Selector (section 2B of the gist.science technical summary of
// "Slow-Fast Inference"): evidence f fused with a positional prior in the closed form
// s = (1 - lambda) f + lambda r, then Top-K positions, ties to the lower position.
//
// One CTA of 1024 threads per unit. The K-th largest score is found by an exact radix
// select on the scores' order-preserving 32-bit keys (digits of 11, 11 and 10 bits, one
// shared-memory histogram pass each); a final ordered pass compacts the chosen positions
// in ascending order with block-wide scans. The fused score uses round-to-nearest
// multiplies and adds with no contraction, so it is bit-reproducible on any IEEE host.
#include "sfi_device.cuh"

namespace sfi {
namespace {

constexpr int NT = kSelectThreads;
constexpr int kWarps = NT / 32;

__device__ __forceinline__ uint32_t order_key(float x)
{
    if (x != x)
        return 0u;
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct Fuse {
    const float *f;  // evidence of the first candidate (position n_sink)
    int n;           // candidates
    float c1, c2, inv_tau;
    __device__ __forceinline__ uint32_t key(int i) const
    {
        const float rt = fminf(1.f, __fmul_rn(static_cast<float>(n - i), inv_tau));
        const float s = __fadd_rn(__fmul_rn(c1, __ldg(f + i)), __fmul_rn(c2, rt));
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

__global__ void __launch_bounds__(NT) select_kernel(const SelectParams p)
{
    __shared__ uint32_t hist[2048];
    __shared__ int scratch[kWarps + 1];
    __shared__ uint32_t sh_digit;
    __shared__ int sh_above;

    pdl_trigger();
    pdl_wait();
    const int u = blockIdx.x;
    const int b = (u / p.n_kv_heads) % p.batch;
    if (p.active && !p.active[b])
        return;
    const int tid = threadIdx.x, lane = tid & 31;
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
    Fuse fz;
    fz.f = p.f + static_cast<size_t>(u) * p.capacity + S;
    fz.n = nC;
    const int tau = p.prior_tau;
    const double Z = (nC >= tau) ? (tau + 1) * 0.5 + static_cast<double>(nC - tau)
                                 : static_cast<double>(nC) * (nC + 1) / (2.0 * tau);
    fz.c1 = __double2float_rn(1.0 - p.lambda);
    fz.c2 = __double2float_rn(p.lambda / Z);
    fz.inv_tau = __double2float_rn(1.0 / tau);

    // ---- radix select of the K-th largest key ------------------------------------------
    uint32_t prefix = 0, pmask = 0;
    int krem = K;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int nbits = pass < 2 ? 11 : 10;
        const int nb = 1 << nbits;
        for (int i = tid; i < nb; i += NT)
            hist[i] = 0u;
        __syncthreads();
        for (int base = 0; base < nC; base += 4 * NT) {
            // four consecutive candidates per thread: their loads are in flight together
            uint32_t k[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = base + 4 * tid + e;
                k[e] = i < nC ? fz.key(i) : 0u;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool part = (base + 4 * tid + e < nC) && ((k[e] & pmask) == prefix);
                const uint32_t digit = (k[e] >> shift) & static_cast<uint32_t>(nb - 1);
                const unsigned act = __ballot_sync(0xffffffffu, part);
                if (part) {
                    const unsigned peers = __match_any_sync(act, digit);
                    if (lane == __ffs(peers) - 1)
                        atomicAdd(&hist[digit], static_cast<uint32_t>(__popc(peers)));
                }
            }
        }
        __syncthreads();
        // thread t owns bins nb-1-per*t ... (descending); find the bin where the count of
        // keys above it first reaches krem
        const int per = nb / NT;
        int mine = 0;
        for (int j = 0; j < per; ++j)
            mine += static_cast<int>(hist[nb - 1 - (per * tid + j)]);
        int total;
        int before = block_exclusive_scan(mine, scratch, &total);
        for (int j = 0; j < per; ++j) {
            const int bin = nb - 1 - (per * tid + j);
            const int h = static_cast<int>(hist[bin]);
            if (before < krem && before + h >= krem) {
                sh_digit = static_cast<uint32_t>(bin);
                sh_above = before;
            }
            before += h;
        }
        __syncthreads();
        prefix |= sh_digit << shift;
        pmask |= static_cast<uint32_t>(nb - 1) << shift;
        krem -= sh_above;
        __syncthreads();
    }
    const uint32_t thr = prefix;  // exact key of the K-th largest score
    const int need_eq = krem;     // how many keys equal to thr are taken (lowest first)

    // ---- ordered compaction ------------------------------------------------------------
    int out_base = 0, eq_base = 0;
    for (int base = 0; base < nC; base += 4 * NT) {
        uint32_t k[4];
        int n_eq = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = base + 4 * tid + e;
            k[e] = i < nC ? fz.key(i) : 0u;
            n_eq += (i < nC && k[e] == thr) ? 1 : 0;
        }
        int tot_eq;
        int eq_before = eq_base + block_exclusive_scan(n_eq, scratch, &tot_eq);
        bool sel[4];
        int n_sel = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = base + 4 * tid + e;
            sel[e] = false;
            if (i < nC) {
                if (k[e] > thr) {
                    sel[e] = true;
                } else if (k[e] == thr) {
                    sel[e] = eq_before < need_eq;
                    ++eq_before;
                }
            }
            n_sel += sel[e] ? 1 : 0;
        }
        int tot_sel;
        int pos = out_base + block_exclusive_scan(n_sel, scratch, &tot_sel);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (sel[e])
                out[pos++] = S + base + 4 * tid + e;
        out_base += tot_sel;
        eq_base += tot_eq;
    }
    if (tid == 0)
        p.sel_cnt[u] = K;
}

}  // namespace

cudaError_t launch_select(const SelectParams &p, cudaStream_t stream)
{
    const cudaError_t e = launch_pdl(select_kernel, dim3(p.n_units), dim3(NT), 0, stream, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace sfi
