// refine.cu -- the Selector's refinements before Top-K (section 2B of the gist.science
// technical summary of "Slow-Fast Inference": Soft-NMS within a head, cross-head
// exclusivity; the prior's key-norm term; the reverse-KL fusion's geometric form) and the
// key norms that term needs. The pages give no formulas: the fp32 recipes below are the
// library's readings, evaluated with round-to-nearest operations in a fixed order (no
// contraction) so that any IEEE host reproduces them bit for bit.
#include "sfi_device.cuh"

namespace sfi {
namespace {

constexpr int kMaxHeads = 16;

// log2 in fp32 from x = 2^e m, m in [1, 2): e + (2/ln 2) atanh(t), t = (m-1)/(m+1), with
// atanh(t) = t (1 + t^2/3 + t^4/5 + ... + t^10/11).
__device__ __forceinline__ float log2_fp32(float x)
{
    if (x != x || x < 0.f)
        return __int_as_float(0x7fc00000);
    if (x == 0.f)
        return -INFINITY;
    if (isinf(x))
        return INFINITY;
    uint32_t u = __float_as_uint(x);
    int e = static_cast<int>((u >> 23) & 0xFFu);
    if (e == 0) {  // subnormal
        u = __float_as_uint(__fmul_rn(x, 4294967296.0f));
        e = static_cast<int>((u >> 23) & 0xFFu) - 32;
    }
    e -= 127;
    const float m = __uint_as_float((u & 0x007FFFFFu) | 0x3F800000u);
    const float t = __fdiv_rn(__fadd_rn(m, -1.0f), __fadd_rn(m, 1.0f));
    const float t2 = __fmul_rn(t, t);
    float s = 0x1.745d18p-4f;
    s = __fadd_rn(__fmul_rn(s, t2), 0x1.c71c72p-4f);
    s = __fadd_rn(__fmul_rn(s, t2), 0x1.24924ap-3f);
    s = __fadd_rn(__fmul_rn(s, t2), 0x1.99999ap-3f);
    s = __fadd_rn(__fmul_rn(s, t2), 0x1.555556p-2f);
    s = __fadd_rn(__fmul_rn(s, t2), 1.0f);
    return __fadd_rn(static_cast<float>(e), __fmul_rn(0x1.715476p+1f, __fmul_rn(t, s)));
}

struct Fused {
    const RefineParams *p;
    int L, nC;
    float c1, c2, inv_tau, lam;
    // fused score of candidate i (position S + i) for the unit u
    __device__ __forceinline__ float at(int u, int i) const
    {
        const int j = p->n_sink + i;
        float rt = fminf(1.f, __fmul_rn(static_cast<float>(nC - i), inv_tau));
        if (p->norm_nu > 0.f && p->key_norms) {
            const float g = fminf(1.f, __fdiv_rn(p->norm_nu,
                                                 __ldg(p->key_norms + static_cast<size_t>(u) * p->capacity + j)));
            rt = __fmul_rn(rt, g);
        }
        const float fj = __ldg(p->f + static_cast<size_t>(u) * p->capacity + j);
        if (!p->geometric)
            return __fadd_rn(__fmul_rn(c1, fj), __fmul_rn(c2, rt));
        const float a = __fmul_rn(c1, log2_fp32(fj));
        float b = 0.f;
        if (p->lambda > 0.0)
            b = __fmul_rn(lam, log2_fp32(__fdiv_rn(__fmul_rn(c2, rt), lam)));
        return p->lambda < 1.0 ? __fadd_rn(a, b) : b;
    }
};

// Soft-NMS: a neighbour's score w suppresses v when it is strictly higher and, with a
// similarity limit delta > 0, close to it: fl32(w - v) <= delta. NaN on either side never
// suppresses.
__device__ __forceinline__ bool nms_suppresses(float w, float v, float delta)
{
    return w > v && (delta <= 0.f || __fadd_rn(w, -v) <= delta);
}

__global__ void __launch_bounds__(256) refine_kernel(const RefineParams p)
{
    pdl_trigger();
    pdl_wait();
    const int lb = blockIdx.y;  // (layer, sequence)
    const int b = lb % p.batch;
    if (p.active && !p.active[b])
        return;
    const int H = p.n_kv_heads;
    const int L = min(p.seq_len[b], p.capacity);
    const int nC = max(0, L - p.n_window - p.n_sink);
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    // fp64 is slow here: one thread computes the constants for the block
    __shared__ float sh_c[5];
    if (threadIdx.x == 0) {
        const int tau = p.prior_tau;
        const double Z = (nC >= tau) ? (tau + 1) * 0.5 + static_cast<double>(nC - tau)
                                     : static_cast<double>(nC) * (nC + 1) / (2.0 * tau);
        sh_c[0] = __double2float_rn(1.0 - p.lambda);
        sh_c[1] = __double2float_rn(p.lambda / Z);
        sh_c[2] = __double2float_rn(1.0 / tau);
        sh_c[3] = __double2float_rn(p.lambda);
        sh_c[4] = H > 1 ? __double2float_rn(static_cast<double>(p.excl_mu) / (H - 1)) : 0.f;
    }
    __syncthreads();
    if (i >= nC)
        return;
    Fused fz;
    fz.p = &p;
    fz.L = L;
    fz.nC = nC;
    fz.c1 = sh_c[0];
    fz.c2 = sh_c[1];
    fz.inv_tau = sh_c[2];
    fz.lam = sh_c[3];
    const int u0 = lb * H;  // units of this (layer, sequence) are u0 .. u0 + H - 1
    float sp[kMaxHeads];
    for (int h = 0; h < H; ++h) {
        const float v = fz.at(u0 + h, i);
        bool dominated = false;
        for (int k = 1; k <= p.nms_radius; ++k) {
            if (i - k >= 0)
                dominated |= nms_suppresses(fz.at(u0 + h, i - k), v, p.nms_delta);
            if (i + k < nC)
                dominated |= nms_suppresses(fz.at(u0 + h, i + k), v, p.nms_delta);
        }
        sp[h] = dominated ? __fmul_rn(p.nms_gamma, v) : v;
    }
    if (p.excl_mu != 0.f && H > 1) {
        const float mu1 = sh_c[4];
        float T = 0.f;
        for (int h = 0; h < H; ++h)
            T = __fadd_rn(T, sp[h]);
        for (int h = 0; h < H; ++h)
            sp[h] = __fadd_rn(sp[h], -__fmul_rn(mu1, __fadd_rn(T, -sp[h])));
    }
    for (int h = 0; h < H; ++h)
        p.refined[static_cast<size_t>(u0 + h) * p.capacity + p.n_sink + i] = sp[h];
}

// One thread per cache row: squares summed in fp32 in dimension order, then sqrt.
__global__ void __launch_bounds__(256) key_norms_kernel(const uint4 *__restrict__ k, float *norms,
                                                        const int32_t *seq_len,
                                                        const uint8_t *active, int batch,
                                                        int n_kv_heads, int capacity,
                                                        int page_size, int n_pages, int max_pages,
                                                        const int32_t *page_table, uint32_t *err)
{
    pdl_trigger();
    pdl_wait();
    const int u = blockIdx.y;
    const int kvh = u % n_kv_heads, b = (u / n_kv_heads) % batch, layer = u / (n_kv_heads * batch);
    if (active && !active[b])
        return;
    const int L = min(seq_len[b], capacity);
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= L)
        return;
    size_t row;
    if (page_size == 0) {
        row = static_cast<size_t>(u) * capacity + j;
    } else {
        const int page = __ldg(page_table + b * max_pages + j / page_size);
        if (page < 0 || page >= n_pages) {
            raise_error(err, 0x1u);
            return;
        }
        row = (static_cast<size_t>(layer * n_pages + page) * n_kv_heads + kvh) * page_size +
              j % page_size;
    }
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        const uint4 w = __ldg(k + row * 16 + c);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float lo = __uint_as_float(ws[q] << 16);
            const float hi = __uint_as_float(ws[q] & 0xFFFF0000u);
            acc = __fadd_rn(acc, __fmul_rn(lo, lo));
            acc = __fadd_rn(acc, __fmul_rn(hi, hi));
        }
    }
    norms[static_cast<size_t>(u) * capacity + j] = __fsqrt_rn(acc);
}

}  // namespace

cudaError_t launch_refine(const RefineParams &p, int n_lb, int max_cand, cudaStream_t stream)
{
    if (p.n_kv_heads > kMaxHeads)
        return cudaErrorInvalidValue;
    dim3 grid((max(max_cand, 1) + 255) / 256, n_lb);
    const cudaError_t e = launch_pdl(refine_kernel, grid, dim3(256), 0, stream, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_key_norms(const void *k, float *norms, const int32_t *seq_len,
                             const uint8_t *active, int n_layers, int batch, int n_kv_heads,
                             int capacity, int page_size, int n_pages, int max_pages,
                             const int32_t *page_table, int max_len, uint32_t *err,
                             cudaStream_t stream)
{
    dim3 grid((max(max_len, 1) + 255) / 256, n_layers * batch * n_kv_heads);
    const cudaError_t e = launch_pdl(key_norms_kernel, grid, dim3(256), 0, stream,
                                     static_cast<const uint4 *>(k), norms, seq_len, active, batch,
                                     n_kv_heads, capacity, page_size, n_pages, max_pages,
                                     page_table, err);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace sfi
