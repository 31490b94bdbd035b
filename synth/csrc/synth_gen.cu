// synth_gen.cu -- GPU twin of synth/gen.py: the same counter-based hash, Irwin-Hall normal,
// bf16 rounding and key-norm models, evaluated on the device so large KV caches can be
// filled in place. Holds none of the SFI method's arithmetic. Every formula here must stay
// bit-identical to the numpy generator (a GPU test compares them).
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kM1 = 0xBF58476D1CE4E5B9ull;
constexpr uint64_t kM2 = 0x94D049BB133111EBull;
constexpr int kD = 128;

__device__ __forceinline__ uint64_t counter(uint64_t stream, uint64_t layer, uint64_t b,
                                            uint64_t head, uint64_t pos, uint64_t d)
{
    return d | (pos << 8) | (head << 32) | (b << 38) | (layer << 46) | (stream << 54);
}

__device__ __forceinline__ uint64_t mix64(uint64_t key, uint64_t ctr)
{
    uint64_t z = key + (ctr + 1ull) * kGamma;
    z = (z ^ (z >> 30)) * kM1;
    z = (z ^ (z >> 27)) * kM2;
    return z ^ (z >> 31);
}

__device__ __forceinline__ float normal_f32(uint64_t h)
{
    const int64_t s = static_cast<int64_t>((h & 0xFFFFull) + ((h >> 16) & 0xFFFFull) +
                                           ((h >> 32) & 0xFFFFull) + ((h >> 48) & 0xFFFFull)) -
                      131070;
    const float x = __fmul_rn(static_cast<float>(s), 1.52587890625e-05f);  // 2^-16, exact
    return __fmul_rn(x, 1.7320508075688772f);                               // fl32(sqrt(3))
}

__device__ __forceinline__ uint16_t f32_to_bf16(float x)
{
    uint32_t u = __float_as_uint(x);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u)
        return 0x7FC0u;
    u += 0x7FFFu + ((u >> 16) & 1u);
    return static_cast<uint16_t>(u >> 16);
}

struct Model {
    int kind;                 // 0 plain, 1 zipf, 2 heavy hitters
    const uint32_t *zthr;     // zipf thresholds [kmax]
    const float *zboost;      // zipf boosts [kmax + 1]
    int zkmax;
    const float *ka;          // heavy-hitter key offset [Ly][Hkv][D]
    const uint32_t *hh_bits;  // heavy-hitter bitmap [units][words]
    int hh_words;
    int n_kv_heads;
    int batch;
};

// One 16-byte chunk (8 dims starting at d0) of the K (stream 0) or V (stream 1) row.
__device__ __forceinline__ uint4 kv_chunk(uint64_t key, int stream, int layer, int b, int head,
                                          int pos, int d0, const Model &m)
{
    float scale = 1.f;
    bool hh = false;
    if (stream == 0 && m.kind == 1) {
        const uint32_t u = static_cast<uint32_t>(mix64(key, counter(3, layer, b, head, pos, 0)) >> 32);
        int lo = 0, hi = m.zkmax;  // first index with u < thr[index], or kmax
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (u < m.zthr[mid])
                hi = mid;
            else
                lo = mid + 1;
        }
        scale = m.zboost[lo];
    } else if (stream == 0 && m.kind == 2) {
        const int unit = (layer * m.batch + b) * m.n_kv_heads + head;
        hh = (m.hh_bits[static_cast<size_t>(unit) * m.hh_words + (pos >> 5)] >> (pos & 31)) & 1u;
    }
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint16_t e[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int d = d0 + 2 * i + j;
            float x = normal_f32(mix64(key, counter(stream, layer, b, head, pos, d)));
            if (m.kind == 1 && stream == 0)
                x = __fmul_rn(x, scale);
            else if (hh)
                x = __fadd_rn(x, m.ka[(layer * m.n_kv_heads + head) * kD + d]);
            e[j] = f32_to_bf16(x);
        }
        w[i] = static_cast<uint32_t>(e[0]) | (static_cast<uint32_t>(e[1]) << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Contiguous cache [Ly][B][Hkv][cap][D]: rows below fill[b] generated, the rest zeroed.
__global__ void fill_contig(uint4 *dst, int stream, int n_layers, int batch, int n_kv_heads,
                            int cap, const int64_t *fill, uint64_t key, Model m)
{
    const uint64_t total = static_cast<uint64_t>(n_layers) * batch * n_kv_heads * cap * 16;
    for (uint64_t i = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
        const int ch = static_cast<int>(i & 15);
        uint64_t row = i >> 4;
        const int pos = static_cast<int>(row % cap);
        row /= cap;
        const int head = static_cast<int>(row % n_kv_heads);
        row /= n_kv_heads;
        const int b = static_cast<int>(row % batch);
        const int layer = static_cast<int>(row / batch);
        dst[i] = pos < fill[b] ? kv_chunk(key, stream, layer, b, head, pos, 8 * ch, m)
                               : make_uint4(0u, 0u, 0u, 0u);
    }
}

// Paged cache [Ly][n_pages][Hkv][16][D] through owner tables (page -> sequence, logical page).
__global__ void fill_paged(uint4 *dst, int stream, int n_layers, int n_pages, int n_kv_heads,
                           const int32_t *owner_b, const int32_t *owner_lp, const int64_t *fill,
                           uint64_t key, Model m)
{
    const uint64_t total = static_cast<uint64_t>(n_layers) * n_pages * n_kv_heads * 16 * 16;
    for (uint64_t i = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
        const int ch = static_cast<int>(i & 15);
        uint64_t row = i >> 4;
        const int slot = static_cast<int>(row & 15);
        row >>= 4;
        const int head = static_cast<int>(row % n_kv_heads);
        row /= n_kv_heads;
        const int page = static_cast<int>(row % n_pages);
        const int layer = static_cast<int>(row / n_pages);
        const int b = owner_b[page];
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (b >= 0) {
            const int pos = owner_lp[page] * 16 + slot;
            if (pos < fill[b])
                v = kv_chunk(key, stream, layer, b, head, pos, 8 * ch, m);
        }
        dst[i] = v;
    }
}

// Rows appended at step t: [steps][Ly][B][Hkv][D], position len0[b] + t.
__global__ void fill_new(uint4 *dst, int stream, int steps, int n_layers, int batch,
                         int n_kv_heads, const int64_t *len0, uint64_t key, Model m)
{
    const uint64_t total = static_cast<uint64_t>(steps) * n_layers * batch * n_kv_heads * 16;
    for (uint64_t i = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
        const int ch = static_cast<int>(i & 15);
        uint64_t row = i >> 4;
        const int head = static_cast<int>(row % n_kv_heads);
        row /= n_kv_heads;
        const int b = static_cast<int>(row % batch);
        row /= batch;
        const int layer = static_cast<int>(row % n_layers);
        const int t = static_cast<int>(row / n_layers);
        dst[i] = kv_chunk(key, stream, layer, b, head, static_cast<int>(len0[b] + t), 8 * ch, m);
    }
}

// Decode queries [steps][Ly][B][Hq][D] (stream 2, position = step), plus qa of the kv group.
__global__ void fill_queries(uint4 *dst, int steps, int n_layers, int batch, int n_q_heads,
                             int group, uint64_t key, const float *qa)
{
    const uint64_t total = static_cast<uint64_t>(steps) * n_layers * batch * n_q_heads * 16;
    for (uint64_t i = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
        const int ch = static_cast<int>(i & 15);
        uint64_t row = i >> 4;
        const int h = static_cast<int>(row % n_q_heads);
        row /= n_q_heads;
        const int b = static_cast<int>(row % batch);
        row /= batch;
        const int layer = static_cast<int>(row % n_layers);
        const int t = static_cast<int>(row / n_layers);
        const int n_kv = n_q_heads / group;
        uint32_t w[4];
        for (int k = 0; k < 4; ++k) {
            uint16_t e[2];
            for (int j = 0; j < 2; ++j) {
                const int d = 8 * ch + 2 * k + j;
                float x = normal_f32(mix64(key, counter(2, layer, b, h, t, d)));
                if (qa)
                    x = __fadd_rn(x, qa[(layer * n_kv + h / group) * kD + d]);
                e[j] = f32_to_bf16(x);
            }
            w[k] = static_cast<uint32_t>(e[0]) | (static_cast<uint32_t>(e[1]) << 16);
        }
        dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

Model make_model(int kind, const uint32_t *zthr, const float *zboost, int zkmax, const float *ka,
                 const uint32_t *hh_bits, int hh_words, int n_kv_heads, int batch)
{
    Model m;
    m.kind = kind;
    m.zthr = zthr;
    m.zboost = zboost;
    m.zkmax = zkmax;
    m.ka = ka;
    m.hh_bits = hh_bits;
    m.hh_words = hh_words;
    m.n_kv_heads = n_kv_heads;
    m.batch = batch;
    return m;
}

int grid_for(uint64_t total)
{
    const uint64_t blocks = (total + 255) / 256;
    return static_cast<int>(blocks < 65536 * 8 ? (blocks ? blocks : 1) : 65536 * 8);
}

}  // namespace

extern "C" {

int synth_fill_contig(void *dst, int stream, int n_layers, int batch, int n_kv_heads, int cap,
                      const int64_t *fill, uint64_t key, int kind, const uint32_t *zthr,
                      const float *zboost, int zkmax, const float *ka, const uint32_t *hh_bits,
                      int hh_words, void *cuda_stream)
{
    const Model m = make_model(kind, zthr, zboost, zkmax, ka, hh_bits, hh_words, n_kv_heads, batch);
    const uint64_t total = static_cast<uint64_t>(n_layers) * batch * n_kv_heads * cap * 16;
    fill_contig<<<grid_for(total), 256, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
        static_cast<uint4 *>(dst), stream, n_layers, batch, n_kv_heads, cap, fill, key, m);
    return static_cast<int>(cudaGetLastError());
}

int synth_fill_paged(void *dst, int stream, int n_layers, int batch, int n_pages, int n_kv_heads,
                     const int32_t *owner_b, const int32_t *owner_lp, const int64_t *fill,
                     uint64_t key, int kind, const uint32_t *zthr, const float *zboost, int zkmax,
                     const float *ka, const uint32_t *hh_bits, int hh_words, void *cuda_stream)
{
    const Model m = make_model(kind, zthr, zboost, zkmax, ka, hh_bits, hh_words, n_kv_heads, batch);
    const uint64_t total = static_cast<uint64_t>(n_layers) * n_pages * n_kv_heads * 256;
    fill_paged<<<grid_for(total), 256, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
        static_cast<uint4 *>(dst), stream, n_layers, n_pages, n_kv_heads, owner_b, owner_lp, fill,
        key, m);
    return static_cast<int>(cudaGetLastError());
}

int synth_fill_new(void *dst, int stream, int steps, int n_layers, int batch, int n_kv_heads,
                   const int64_t *len0, uint64_t key, int kind, const uint32_t *zthr,
                   const float *zboost, int zkmax, const float *ka, const uint32_t *hh_bits,
                   int hh_words, void *cuda_stream)
{
    const Model m = make_model(kind, zthr, zboost, zkmax, ka, hh_bits, hh_words, n_kv_heads, batch);
    const uint64_t total = static_cast<uint64_t>(steps) * n_layers * batch * n_kv_heads * 16;
    fill_new<<<grid_for(total), 256, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
        static_cast<uint4 *>(dst), stream, steps, n_layers, batch, n_kv_heads, len0, key, m);
    return static_cast<int>(cudaGetLastError());
}

int synth_fill_queries(void *dst, int steps, int n_layers, int batch, int n_q_heads, int group,
                       uint64_t key, const float *qa, void *cuda_stream)
{
    const uint64_t total = static_cast<uint64_t>(steps) * n_layers * batch * n_q_heads * 16;
    fill_queries<<<grid_for(total), 256, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
        static_cast<uint4 *>(dst), steps, n_layers, batch, n_q_heads, group, key, qa);
    return static_cast<int>(cudaGetLastError());
}

}  // extern "C"

// ---------------------------------------------------------------------------------------
// Heavy-hitter drift: rewrite the K rows of listed positions of a contiguous cache
// [Ly][B][Hkv][cap][D] with their new planted / plain content (V rows do not change).
// pos, planted: [units][m] (pos < 0 = unused slot).
namespace {

__global__ void rewrite_k(uint4 *dst, int n_units, int m, const int32_t *pos,
                          const uint8_t *planted, int batch, int n_kv_heads, int cap,
                          uint64_t key, const float *ka)
{
    const uint64_t total = static_cast<uint64_t>(n_units) * m * 16;
    for (uint64_t i = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
        const int ch = static_cast<int>(i & 15);
        const uint64_t slot = i >> 4;
        const int unit = static_cast<int>(slot / m);
        const int p = pos[slot];
        if (p < 0 || p >= cap)
            continue;
        const int head = unit % n_kv_heads;
        const int b = (unit / n_kv_heads) % batch;
        const int layer = unit / (n_kv_heads * batch);
        uint32_t w[4];
        for (int k = 0; k < 4; ++k) {
            uint16_t e[2];
            for (int j = 0; j < 2; ++j) {
                const int d = 8 * ch + 2 * k + j;
                float x = normal_f32(mix64(key, counter(0, layer, b, head, p, d)));
                if (planted[slot])
                    x = __fadd_rn(x, ka[(layer * n_kv_heads + head) * kD + d]);
                e[j] = f32_to_bf16(x);
            }
            w[k] = static_cast<uint32_t>(e[0]) | (static_cast<uint32_t>(e[1]) << 16);
        }
        dst[(static_cast<uint64_t>(unit) * cap + p) * 16 + ch] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

}  // namespace

extern "C" int synth_rewrite_k(void *dst, int n_units, int m, const int32_t *pos,
                               const uint8_t *planted, int batch, int n_kv_heads, int cap,
                               uint64_t key, const float *ka, void *cuda_stream)
{
    const uint64_t total = static_cast<uint64_t>(n_units) * m * 16;
    rewrite_k<<<grid_for(total), 256, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
        static_cast<uint4 *>(dst), n_units, m, pos, planted, batch, n_kv_heads, cap, key, ka);
    return static_cast<int>(cudaGetLastError());
}
