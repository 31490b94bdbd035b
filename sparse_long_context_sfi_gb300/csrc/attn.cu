// attn.cu -- GQA decode attention for the SFI slow step (dense over the whole KV cache,
// emitting the Selector's evidence) and fast step (packed sparse memory + recent window).
//
// Slow step: the blog "How SFI Works" (dense attention over the full cache) and section 2A
// of the gist.science technical summary ("Slow Steps"). Fast step: the same attention over
// the sparse state of section 2A (sinks + selected memory + sliding window), read as
// section 3 describes: packed sink/selected rows streamed contiguously, recent tokens
// straight from the (possibly paged) cache.
//
// Design (one kernel template for both steps):
//   * Persistent CTAs, one per SM. The tiles of all units (layer, sequence, kv head) are
//     concatenated; CTA c streams the contiguous tile range [c T / P, (c+1) T / P). Units
//     cut by a range boundary are merged by the last CTA to finish them (atomic ticket, no
//     waiting); a unit inside one range is written directly.
//   * Warp 0 issues TMA loads of 128-row K and V tiles (128-byte swizzle) into a 3-stage
//     shared-memory ring. Warp 1 issues tcgen05 UMMAs: S^T = K Q^T (M = 128 positions,
//     N = 16 = query heads padded) and O^T = V^T P^T (M = 128 dims, V read MN-major),
//     accumulating in TMEM. Warps 2-5 run the online softmax one position per thread
//     (tcgen05.ld of S^T), write P^T as bf16 and accumulate O^T one dim per thread.
//   * P carries about 16 significant bits at no extra MMA: head h's weight p goes to operand
//     row h as bf16(p) and its remainder p - bf16(p) to the otherwise unused row G + h, so
//     O^T columns h and G + h hold the two parts and their sum is taken at accumulation.
//     (A bf16-only P errs by up to 2^-9 of a weight, which near-cancelling outputs of two
//     competing heavy positions turn into absolute errors above 2e-3.)
//   * Every wait is bounded; a wait that gives up flags SFI_DEVERR_TIMEOUT, drains the
//     CTA's copies and MMAs, frees TMEM and returns.
#include <math.h>
#include <cstddef>

#include <mutex>

#include "sfi_device.cuh"

namespace sfi {
namespace {
// Remote shared-memory stores whose completion is counted in bytes on the receiving CTA's
// mbarrier (st.async ... mbarrier::complete_tx): no separate arrive or release fence.
__device__ __forceinline__ void st_async_f32x4(uint32_t addr, float a, float b, float c, float d, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
                 :: "r"(addr), "f"(a), "f"(b), "f"(c), "f"(d), "r"(bar) : "memory");
}
__device__ __forceinline__ void st_async_f32x2(uint32_t addr, float a, float b, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
                 :: "r"(addr), "f"(a), "f"(b), "r"(bar) : "memory");
}
__device__ __forceinline__ void st_async_f32(uint32_t addr, float a, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];"
                 :: "r"(addr), "f"(a), "r"(bar) : "memory");
}

constexpr int kChunkBytes = kTile * 128;       // 128 rows x 128 B: one 64-dim half of a tile
constexpr int kStageBytes = 4 * kChunkBytes;   // K[0:64), K[64:128), V[0:64), V[64:128)
constexpr int kOpRows = 16;                    // UMMA N: query heads padded to 16 rows
constexpr int kOpChunk = kOpRows * 128;        // one 64-element K-chunk of Q^T or P^T
constexpr int kOpBytes = 2 * kOpChunk;
static_assert(2 * 8 <= kOpRows, "P^T needs 2 G operand rows (bf16 part and remainder)");
constexpr uint32_t kTmemCols = 64;             // S^T x2 (cols 0, 16), O^T x2 (cols 32, 48)

constexpr int kQOff = kStages * kStageBytes;
constexpr int kPOff = kQOff + 2 * kOpBytes;
constexpr int kCtrlOff = kPOff + 2 * kOpBytes;

constexpr int kMetaRing = 8;    // slots of the tile-metadata ring (see Ctrl)
constexpr int kFlagFirst = 1;   // first tile of a segment (a unit's tiles inside one CTA)
constexpr int kFlagLast = 2;    // last tile of a segment

struct TileMeta {
    int unit;
    int tile;
    int flags;
    int pad;
    uint32_t valid[4];          // bit r: row r of the tile holds a real position
};

struct Ctrl {
    // Ring barriers per stage, separate for the K and the V half: K is free again once the
    // score MMA has read it, V only after the P.V MMA, so the next tile's K can land early.
    uint64_t fullK[kStages], fullV[kStages], emptyK[kStages], emptyV[kStages];
    uint64_t s_full[2], s_free[2], p_full[2], o_full[2], o_free[2], q_free[2];
    uint64_t gsync;             // softmax-group barrier (one arrive per warp)
    uint64_t drain;             // MMA drain on exit
    uint64_t unit_meta;         // clustered: the unit's length and activity are known
    uint64_t cl_ready;          // clustered: every CTA of the cluster has its partial in place
    uint64_t q_full;            // clustered: the query has landed
    // Tile metadata (unit, flags, row mask) in a ring of its own, one barrier per slot: the
    // producer publishes tile j only after the score MMA of tile j - 3, which the MMA issued
    // after the softmax had read tile j - 5's metadata, so at most tiles j - 4 .. j - 1 are
    // unread: kMetaRing >= 5 slots never collide, and a slot's barrier is never two phases
    // ahead of the softmax waiting on it.
    uint64_t meta_full[kMetaRing];
    TileMeta meta[kMetaRing];
    float red_max[2][4][8];
    float red_sum[4][8];
    uint32_t tmem_base;
    int abort;
    int last_flag;
    int cl_live;                // clustered: the unit is active and its length valid
    int P;
    long long T, TL, g0, g1;
    int nt[kMaxBatch];
    int pre[kMaxBatch];
    int len[kMaxBatch];
};

constexpr int kSmemBytes = kCtrlOff + static_cast<int>(sizeof(Ctrl)) + 1024;

// The mbarriers of Ctrl, fullK[0] through meta_full[kMetaRing - 1], lie back to back; the
// softmax-group ones (s_free, p_full, o_free, gsync) expect one arrival per softmax warp,
// the others one. Set up in one plain loop over that range.
constexpr int kNBars = static_cast<int>(
    (offsetof(Ctrl, meta_full) + kMetaRing * sizeof(uint64_t) - offsetof(Ctrl, fullK)) / sizeof(uint64_t));
constexpr int bar_index(size_t off) { return static_cast<int>((off - offsetof(Ctrl, fullK)) / sizeof(uint64_t)); }
constexpr uint64_t kFourArrivals = (3ull << bar_index(offsetof(Ctrl, s_free))) |
                                   (3ull << bar_index(offsetof(Ctrl, p_full))) |
                                   (3ull << bar_index(offsetof(Ctrl, o_free))) |
                                   (1ull << bar_index(offsetof(Ctrl, gsync)));
static_assert(kNBars == 4 * kStages + 12 + 5 + kMetaRing && kNBars <= 64, "mbarriers of Ctrl");

// Warp-wide max of non-NaN floats in one redux: the float bits as a signed integer, with the
// magnitude bits of negatives flipped, order like the floats (-inf lowest, -0 below +0).
__device__ __forceinline__ float warp_max(float x)
{
    int k = __float_as_int(x);
    k ^= (k >> 31) & 0x7fffffff;
    int m = __reduce_max_sync(0xffffffffu, k);
    m ^= (m >> 31) & 0x7fffffff;
    return __int_as_float(m);
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Barrier over the four softmax warps through an mbarrier, so it can give up.
__device__ __forceinline__ bool group_sync(Ctrl &c, uint32_t &phase, int lane)
{
    __syncwarp();
    if (lane == 0)
        mbar_arrive(&c.gsync);
    const bool ok = mbar_wait(&c.gsync, phase & 1u, &c.abort);
    ++phase;
    return ok;
}

__device__ __forceinline__ void fail(Ctrl &c, uint32_t *err)
{
    c.abort = 1;
    raise_error(err, 0x4u);  // SFI_DEVERR_TIMEOUT
}

// Set rows [r0, r1) of a 128-row validity mask kept in four registers.
__device__ __forceinline__ uint32_t word_bits(int r0, int r1, int w)
{
    const int lo = min(max(r0 - 32 * w, 0), 32), hi = min(max(r1 - 32 * w, 0), 32);
    if (hi <= lo)
        return 0u;
    const uint32_t upto = hi == 32 ? 0xffffffffu : ((1u << hi) - 1u);
    return upto & ~((1u << lo) - 1u);
}

__device__ __forceinline__ void mask_rows(uint32_t (&v)[4], int r0, int r1)
{
#pragma unroll
    for (int w = 0; w < 4; ++w)
        v[w] |= word_bits(r0, r1, w);
}

// 2^x with the hardware approximation (PTX ex2.approx.ftz: relative error ~2^-22,
// subnormal results flushed to zero; 2^-inf = 0). Used for the softmax weights, which are
// rounded to bf16 for the O MMA anyway.
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// a[i] for a small register array without dynamic indexing (which would move the array to
// local memory)
template <int G>
__device__ __forceinline__ float pick(const float (&a)[G], int i)
{
    float v = a[0];
#pragma unroll
    for (int h = 1; h < G; ++h)
        v = (i == h) ? a[h] : v;
    return v;
}

template <int G>
__device__ __forceinline__ void store_out(const AttnParams &p, int u, int d, const float (&o)[G])
{
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const size_t idx = (static_cast<size_t>(u) * G + h) * kHeadDim + d;
        if (p.out_fp32)
            static_cast<float *>(p.out)[idx] = o[h];
        else
            static_cast<__nv_bfloat16 *>(p.out)[idx] = __float2bfloat16_rn(o[h]);
    }
}

template <int G, bool DENSE, bool CL>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
                const __grid_constant__ CUtensorMap tm_vc, const AttnParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Ctrl &c = *reinterpret_cast<Ctrl *>(smem + kCtrlOff);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = p.batch, Hkv = p.n_kv_heads;

    // ---- set-up touching no global memory: overlaps the previous kernel's tail ----------
    pdl_trigger();
    // the tensor maps' descriptors, fetched while the barriers are set up
    if (warp == 1 && lane < (DENSE ? 3 : 5))
        tma_prefetch_map(lane == 0 ? &tm_k : lane == 1 ? &tm_v : lane == 2 ? &tm_q
                                    : lane == 3 ? &tm_kc : &tm_vc);
    // CL: the clustered fast step, compiled as its own instance (launched only with
    // p.cluster > 1), so neither instance carries the other's code paths; with DENSE, the
    // dense step with the fused append
    constexpr bool clustered = !DENSE && CL;
    // fused append (the fast step with p.k_new set; the dense step's instance with CL set):
    // the new K/V rows are written at position seq_len[b] and attended, and the last CTA
    // advances seq_len. The plain dense instance carries none of the append's code.
    const bool fused = DENSE ? CL : (p.k_new != nullptr);
    // Clustered fast step: this CTA's unit and its static slice [cl_t0, cl_t0 + cl_n) of the
    // unit's tiles (the MMA and softmax roles iterate over the whole slice; a unit found
    // inactive only gets empty tiles and no output). Producer state: the unit's packed row
    // count cl_rows and packed sinks cl_ns, and cl_i, the next tile of the slice to publish.
    int cl_u = 0, cl_t0 = 0, cl_n = 0, cl_rows = 0, cl_ns = 0, cl_i = 0, cl_pre = 0;
    if (clustered) {
        cl_u = static_cast<int>(blockIdx.x) / p.cluster;
        const int rank = static_cast<int>(blockIdx.x) % p.cluster;
        cl_t0 = rank * p.tiles_per_unit / p.cluster;
        cl_n = (rank + 1) * p.tiles_per_unit / p.cluster - cl_t0;
        // tiles requested before the wait: those of packed rows only, at most kStages
        cl_pre = max(0, min(min(kStages, cl_n), 64 * p.n_cbox / kTile - cl_t0));
    }
    if (warp == 0) {
        // the barriers of the set-up, spread over the warp's lanes (its fence then publishes
        // them all)
        uint64_t *bars = &c.fullK[0];
        for (int idx = lane; idx < kNBars; idx += 32)
            mbar_init(bars + idx, ((kFourArrivals >> idx) & 1ull) ? 4u : 1u);
        mbar_fence_init();
        __syncwarp();
        // clustered: the query's bytes, requested right after the wait
        if (clustered && lane == 0)
            mbar_arrive_expect_tx(&c.q_full, 2u * G * 128u);
    }
    if (tid == 0) {
        c.abort = 0;
        c.cl_live = 0;
    }
    if (warp == 1) {
        tmem_alloc(&c.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    // Q^T and P^T operands: rows >= G stay zero for the whole kernel.
    for (int i = tid; i < 4 * kOpBytes / 16; i += kAttnThreads)
        reinterpret_cast<uint4 *>(smem + kQOff)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    // Clustered fast step: one unit per cluster, its tiles split evenly over the cluster's
    // CTAs, which merge their partials through distributed shared memory. The peers need
    // only this CTA's mbarrier initialisation, which fence.mbarrier_init has published, so
    // the cluster arrival is relaxed; the CTA barrier publishes the TMEM base.
    if (clustered) {
        // arrive now, wait only before the first access to a peer's shared memory (the merge)
        tc_fence_before();
        cluster_arrive_relaxed();
        __syncthreads();
        tc_fence_after();
    }
    // The packed memory is complete before this launch starts (sfi_compact and
    // sfi_select let their dependents start only after their writes), so the slice's
    // first tiles of packed rows are requested before the wait on the preceding grid: every
    // box of them, since the unit's packed row count is known only after the wait (rows
    // past it are masked then). Their arrival on full lets the score MMAs start as soon as
    // the query lands. A softmax warp issues them (it is idle until the first scores), so
    // the producer warp reaches the wait, and the query load, without them.
    if (clustered && warp == 2) {
        const int h2 = lane >> 4, j16 = lane & 15;
        for (int i = 0; i < cl_pre; ++i) {
            if (lane == 0) {
                mbar_arrive_expect_tx(&c.fullK[i], 2u * 2u * 64u * 128u +
                                                       ((p.test_stall && blockIdx.x == 0 && i == 0) ? 16u : 0u));
                mbar_arrive_expect_tx(&c.fullV[i], 2u * 2u * 64u * 128u);
            }
            __syncwarp();
            if (j16 < 4) {
                const int k = ((cl_t0 + i) * kTile + 64 * h2) >> 6;
                const int kv = j16 >> 1, half = j16 & 1;
                tma_load_2d(smem + i * kStageBytes + kv * 2 * kChunkBytes + half * kChunkBytes +
                                64 * h2 * 128,
                            kv ? &tm_vc : &tm_kc, kv ? &c.fullV[i] : &c.fullK[i], 64 * half,
                            cl_u * p.comp_cap + 64 * k);
            }
        }
    }

    // Clustered fast step: the unit's query rows and (fused append) its new K/V rows are
    // read only after the wait, as they may come from the preceding kernel; prefetching them
    // into L2 now is harmless either way (L2 is where the preceding kernel's writes land)
    // and takes a DRAM round trip off the path after the wait when they were written
    // earlier. (Done for the tile-range step's first unit as well, it was measured slower:
    // finding that unit before the wait costs the late CTAs more than the prefetch saves.)
    if (clustered && warp == 3 && lane == 0) {
        tma_prefetch_l2_2d(&tm_q, 0, cl_u * G);
        tma_prefetch_l2_2d(&tm_q, 64, cl_u * G);
        if (fused) {
            bulk_prefetch_l2(static_cast<const char *>(p.k_new) + static_cast<size_t>(cl_u) * 256, 256u);
            bulk_prefetch_l2(static_cast<const char *>(p.v_new) + static_cast<size_t>(cl_u) * 256, 256u);
        }
    }

    // Tile t of the slice in ring stage i % kStages (producer warp, clustered): its row mask
    // is written and published on meta_full (what the softmax waits for), and with `issue`
    // its boxes are requested on full (what the MMA waits for): the packed rows below
    // cl_rows in 64-row boxes, and with `win` the window boxes of a sequence of length L
    // whose window starts at ws (wpg: the page of this lane's window box, paged cache).
    auto cl_tile = [&](int i, int t, bool win, int L, int ws, int wpg, bool issue) -> bool {
        const int s = i % kStages;
        const int h2 = lane >> 4, j16 = lane & 15, op = lane & 3;
        const int R = t * kTile + 64 * h2;
        const CUtensorMap *map = nullptr;
        int y = 0, row0 = 0, rows = 0, kv = 0, half = 0;
        uint32_t valid[4] = {0u, 0u, 0u, 0u};
        if (R < 64 * p.n_cbox) {
            const int k = R >> 6;
            const int vr = max(0, min(64, cl_rows - 64 * k));
            if (vr > 0 && j16 < 4) {
                kv = j16 >> 1;
                half = j16 & 1;
                map = kv ? &tm_vc : &tm_kc;
                y = cl_u * p.comp_cap + 64 * k;
                row0 = 64 * h2;
                rows = 64;
                if (j16 == 0)
                    mask_rows(valid, row0, row0 + vr);
            }
        } else if (win) {
            const int q = j16 >> 2;
            const int j = (R + 16 * q - 64 * p.n_cbox) >> 4;
            const int rr0 = 64 * h2 + 16 * q;
            if (j < p.n_wbox && p.page_size == 0) {
                const int p0 = ws + 16 * j;
                const int vr = max(0, min(16, L - p0));
                if (vr > 0) {
                    kv = op >> 1;
                    half = op & 1;
                    map = kv ? &tm_v : &tm_k;
                    y = cl_u * p.capacity + p0;
                    row0 = rr0;
                    rows = 16;
                    if (op == 0)
                        mask_rows(valid, rr0, rr0 + vr);
                }
            } else if (j < p.n_wbox) {
                const int lp = (ws >> 4) + j;
                const int r0 = max(ws - lp * 16, 0), r1 = min(L - lp * 16, 16);
                if (r1 > r0) {
                    const int b = (cl_u / Hkv) % B, layer = cl_u / (Hkv * B), kvh = cl_u % Hkv;
                    const int page = p.n_wbox <= 32 ? wpg : __ldg(p.page_table + b * p.max_pages + lp);
                    if (page < 0 || page >= p.n_pages) {
                        if (op == 0)
                            raise_error(p.err, 0x1u);  // SFI_DEVERR_PAGE_RANGE
                    } else {
                        kv = op >> 1;
                        half = op & 1;
                        map = kv ? &tm_v : &tm_k;
                        y = ((layer * p.n_pages + page) * Hkv + kvh) * 16;
                        row0 = rr0;
                        rows = 16;
                        if (op == 0)
                            mask_rows(valid, rr0 + r0, rr0 + r1);
                    }
                }
            }
        }
        uint32_t vw[4];
#pragma unroll
        for (int w = 0; w < 4; ++w)
            vw[w] = __reduce_or_sync(0xffffffffu, valid[w]);
        // test hook: CTA 0's first tile expects 16 bytes that never come (sfi_test_inject_stall)
        const uint32_t bytes_k =
            __reduce_add_sync(0xffffffffu, kv == 0 ? static_cast<uint32_t>(rows) * 128u : 0u) +
            ((p.test_stall && blockIdx.x == 0 && i == 0) ? 16u : 0u);
        const uint32_t bytes_v =
            __reduce_add_sync(0xffffffffu, kv == 1 ? static_cast<uint32_t>(rows) * 128u : 0u);
        uint8_t *dst = smem + s * kStageBytes + kv * 2 * kChunkBytes + half * kChunkBytes + row0 * 128;
        if (lane == 0) {
            TileMeta &mt = c.meta[i % kMetaRing];
            mt.unit = cl_u;
            mt.tile = t;
            mt.flags = (i == 0 ? kFlagFirst : 0) | (i == cl_n - 1 ? kFlagLast : 0);
#pragma unroll
            for (int w = 0; w < 4; ++w)
                mt.valid[w] = vw[w];
            mbar_arrive(&c.meta_full[i % kMetaRing]);  // releases the metadata
            if (issue)
                mbar_arrive_expect_tx(&c.fullK[s], bytes_k);
        }
        __syncwarp();
        if (!issue)
            return true;
        if (rows > 0 && kv == 0)
            tma_load_2d(dst, map, &c.fullK[s], 64 * half, y);
        // the V half: free once the P.V MMA of this stage's previous tile is done
        bool okv = true;
        if (lane == 0)
            okv = mbar_wait(&c.emptyV[s], ((i / kStages) & 1) ^ 1, &c.abort);
        if (!__shfl_sync(0xffffffffu, okv ? 1 : 0, 0))
            return false;
        if (lane == 0)
            mbar_arrive_expect_tx(&c.fullV[s], bytes_v);
        __syncwarp();
        if (rows > 0 && kv == 1)
            tma_load_2d(dst, map, &c.fullV[s], 64 * half, y);
        return true;
    };
    // ---- tile space: per-sequence tile counts and this CTA's range --------------------
    long long g0 = 0, g1 = 0;
    int n_tiles = 0;
    // exclusive prefix sum of the per-sequence tile counts c.nt, one warp (each lane sums a
    // contiguous run of up to 8 sequences, batch <= 256, then a warp scan), and this CTA's
    // stream-K range: equal contiguous tile ranges (balances ragged lengths and unit counts
    // that are not a multiple of the CTA count); all threads, ends with a CTA barrier
    auto tile_space = [&]() {
        if (warp == 0) {
            const int per = (B + 31) / 32, b0 = lane * per;
            int run = 0;
            for (int j = 0; j < per; ++j)
                run += (b0 + j < B) ? c.nt[b0 + j] : 0;
            int incl = run;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += y;
            }
            int acc = incl - run;
            for (int j = 0; j < per && b0 + j < B; ++j) {
                c.pre[b0 + j] = acc * Hkv;
                acc += c.nt[b0 + j];
            }
            const int total = __shfl_sync(0xffffffffu, incl, 31);
            if (lane == 0) {
                c.TL = static_cast<long long>(total) * Hkv;
                c.T = c.TL * p.n_layers;
                c.P = static_cast<int>(c.T < gridDim.x ? c.T : gridDim.x);
                const long long P = c.P > 0 ? c.P : 1;
                c.g0 = static_cast<long long>(blockIdx.x) * c.T / P;
                c.g1 = static_cast<long long>(blockIdx.x + 1) * c.T / P;
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // CTAs beyond the tile count (short contexts) only tear down.
        g0 = c.g0;
        g1 = c.g1;
        n_tiles = static_cast<int>(blockIdx.x) < c.P ? static_cast<int>(g1 - g0) : 0;
    };
    // the first tile of the range: (layer, sequence, kv head, tile of the unit); the
    // sequence is the first with tiles whose range ends past r, found 32 sequences per step
    // by a warp ballot (whole warp)
    auto first_tile = [&](int &layer, int &b, int &kvh, int &t) {
        layer = static_cast<int>(g0 / c.TL);
        const int r = static_cast<int>(g0 - static_cast<long long>(layer) * c.TL);
        b = B - 1;
        for (int b0 = 0; b0 < B; b0 += 32) {
            const int bb = b0 + lane;
            const unsigned m = __ballot_sync(
                0xffffffffu, bb < B && c.nt[bb] > 0 && c.pre[bb] + Hkv * c.nt[bb] > r);
            if (m) {
                b = b0 + __ffs(m) - 1;
                break;
            }
        }
        kvh = (r - c.pre[b]) / c.nt[b];
        t = (r - c.pre[b]) - kvh * c.nt[b];
    };
    // Sparse step over tile ranges: every active sequence has tiles_per_unit tiles, so the
    // tile space depends only on `active` (an input complete at launch) and is laid out before
    // the wait on the preceding grid; the lengths read after it only decide which units give
    // output (c.len[b] <= 0: none). Nothing else is read before the wait: loading the first
    // unit's packed counts, or requesting its first packed tiles, there as well was measured
    // slower on the ragged batch-32 workload (by 2.1 and 0.4 us): the CTAs that enter last
    // carry their set-up on the critical path.
    if (!clustered && !DENSE) {
        for (int b = tid; b < B; b += kAttnThreads)
            c.nt[b] = (p.active ? p.active[b] : 1) ? p.tiles_per_unit : 0;
        __syncthreads();
        tile_space();
    }
    pdl_wait();
    if (!clustered && !DENSE) {
        for (int b = tid; b < B; b += kAttnThreads) {
            const int L0 = p.seq_len[b];
            const int L = fused ? L0 + 1 : L0;  // with the fused append: the new row included
            int act = c.nt[b] > 0;
            if (act && (L0 < 0 || L0 > p.max_len || L > p.capacity)) {
                raise_error(p.err, 0x8u);  // SFI_DEVERR_LENGTH
                act = 0;
            }
            c.len[b] = act ? L : 0;
        }
        __syncthreads();
    } else if (!clustered) {
        for (int b = tid; b < B; b += kAttnThreads) {
            const int L0 = p.seq_len[b];
            const int L = fused ? L0 + 1 : L0;
            int act = p.active ? p.active[b] : 1;
            if (act && (L0 < 0 || L0 > p.max_len || L > p.capacity)) {
                raise_error(p.err, 0x8u);  // SFI_DEVERR_LENGTH
                act = 0;
            }
            c.nt[b] = (act && L > 0) ? (L + kTile - 1) / kTile : 0;
            c.len[b] = L;
        }
        __syncthreads();
        tile_space();
    } else {
        n_tiles = cl_n;
        g0 = cl_t0;
        g1 = g0 + n_tiles;
    }
    const uint32_t tmem = c.tmem_base;

    if (warp == 0 && clustered) {
        // ========================= TMA producer, clustered fast step =======================
        // After the wait: the query first (its own barrier, armed before the wait: it may come
        // from the preceding kernel), then the unit's length, activity and packed counts in
        // one round, then the row masks of the tiles requested before the wait and the rest of
        // the slice; the window tile gets the new row written into the cache (fused append)
        // before its boxes are issued.
        if (lane < 2)
            tma_load_2d(smem + kQOff + lane * kOpChunk, &tm_q, &c.q_full, 64 * lane, cl_u * G);
        const int layer = cl_u / (Hkv * B), b = (cl_u / Hkv) % B, kvh = cl_u % Hkv;
        int v = 0;
        if (lane == 0)
            v = p.seq_len[b];
        else if (lane == 1)
            v = p.active ? p.active[b] : 1;
        else if (lane == 2)
            v = __ldg(p.comp_rows + cl_u);
        else if (lane == 3)
            v = __ldg(p.sel_cnt + cl_u);
        const int L0 = __shfl_sync(0xffffffffu, v, 0);
        const int act = __shfl_sync(0xffffffffu, v, 1);
        const int v2 = __shfl_sync(0xffffffffu, v, 2), v3 = __shfl_sync(0xffffffffu, v, 3);
        cl_rows = max(0, min(v2, p.comp_cap));
        cl_ns = max(0, cl_rows - max(0, v3));
        const int L = fused ? L0 + 1 : L0;  // with the fused append: the new row included
        bool live = act != 0;
        if (live && (L0 < 0 || L0 > p.max_len || L > p.capacity)) {
            if (lane == 0)
                raise_error(p.err, 0x8u);  // SFI_DEVERR_LENGTH
            live = false;
        }
        live = live && L > 0;
        const int ws = max(cl_ns, L - p.n_window);
        // paged: the page of every window box, one per lane (up to 32 boxes)
        const bool wpf = p.page_size != 0 && p.n_wbox <= 32;
        int wpage = 0;
        if (live && wpf) {
            const int lp = (ws >> 4) + lane;
            wpage = (lane < p.n_wbox && lp * 16 < L) ? __ldg(p.page_table + b * p.max_pages + lp) : 0;
        }
        // The tile of this slice that holds the new row (position L - 1), if any: the window
        // tile that reads it; a row outside the window (only in an inconsistent sparse state)
        // is still written once, by the unit's first tile.
        int app = -1, jn = 0;
        if (fused && live) {
            jn = p.page_size == 0 ? ((L - 1 - ws) >> 4) : (((L - 1) >> 4) - (ws >> 4));
            const int t_new = L - 1 >= ws ? (64 * p.n_cbox + 16 * jn) / kTile : 0;
            app = (t_new >= cl_t0 && t_new < cl_t0 + cl_n) ? t_new : -1;
        }
        if (lane == 0) {
            c.cl_live = live ? 1 : 0;
            mbar_arrive(&c.unit_meta);
        }
        // Fused append: the new K and V rows go to position L - 1, 16 bytes per lane (lanes
        // 0-15 K, 16-31 V); each lane fences its write against the async proxy and the warp
        // synchronises before the box covering the row is issued.
        auto append_new_row = [&]() {
            const int pos = L - 1;
            long long row = static_cast<long long>(cl_u) * p.capacity + pos;
            bool good = true;
            if (p.page_size != 0) {
                int page = __shfl_sync(0xffffffffu, wpage, max(0, min(jn, 31)));
                if (!wpf || jn < 0 || jn >= p.n_wbox)
                    page = __ldg(p.page_table + b * p.max_pages + (pos >> 4));
                good = page >= 0 && page < p.n_pages;
                if (!good && lane == 0)
                    raise_error(p.err, 0x1u);  // SFI_DEVERR_PAGE_RANGE
                row = ((static_cast<long long>(layer) * p.n_pages + page) * Hkv + kvh) * 16 + (pos & 15);
            }
            if (good) {
                const int kvsel = lane >> 4, chunk = lane & 15;
                const uint4 x = static_cast<const uint4 *>(kvsel ? p.v_new : p.k_new)
                    [static_cast<size_t>(cl_u) * 16 + chunk];
                static_cast<uint4 *>(kvsel ? p.v_cache : p.k_cache)[row * 16 + chunk] = x;
                fence_proxy_async_global();
            }
            __syncwarp();
        };
        // masks of the tiles requested before the wait (packed rows only)
        for (; cl_i < cl_pre; ++cl_i)
            cl_tile(cl_i, cl_t0 + cl_i, false, 0, 0, 0, false);
        if (app >= 0 && app < cl_t0 + cl_i)   // its tile was requested before the wait
            append_new_row();
        bool ok = true;
        for (; cl_i < cl_n; ++cl_i) {
            const int st = cl_i % kStages, t = cl_t0 + cl_i;
            if (lane == 0)
                ok = mbar_wait(&c.emptyK[st], ((cl_i / kStages) & 1) ^ 1, &c.abort);
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
                if (lane == 0)
                    fail(c, p.err);
                break;
            }
            const bool has_win = live && (t + 1) * kTile > 64 * p.n_cbox;
            int wpg = 0;
            if (has_win && wpf) {
                const int jl = (t * kTile + 64 * (lane >> 4) + 16 * ((lane & 15) >> 2) -
                                64 * p.n_cbox) >> 4;
                wpg = __shfl_sync(0xffffffffu, wpage, jl & 31);
            }
            if (t == app)
                append_new_row();
            if (!cl_tile(cl_i, t, has_win, L, ws, wpg, true)) {
                // its K half may be in flight; its V half was never requested: complete that
                // phase with a bare arrival so the drain below does not wait for it
                if (lane == 0) {
                    mbar_arrive(&c.fullV[st]);
                    fail(c, p.err);
                }
                ++cl_i;
                break;
            }
        }
        // Never leave a copy in flight into shared memory we are about to give up.
        if (lane == 0) {
            for (int j = max(0, cl_i - kStages); j < cl_i; ++j) {
                mbar_wait(&c.fullK[j % kStages], (j / kStages) & 1, nullptr);
                mbar_wait(&c.fullV[j % kStages], (j / kStages) & 1, nullptr);
            }
            mbar_wait(&c.q_full, 0, nullptr);
        }
        // Fused append: the last CTA of the grid to get here advances the lengths.
        if (fused) {
            int is_last = 0;
            if (lane == 0)
                is_last = atomic_add_acq_rel_gpu(p.append_counter, 1) == static_cast<int>(gridDim.x) - 1;
            if (__shfl_sync(0xffffffffu, is_last, 0)) {
                int32_t *len = const_cast<int32_t *>(p.seq_len);
                for (int bb = lane; bb < B; bb += 32) {
                    const int Lb = len[bb];
                    const int ab = p.active ? p.active[bb] : 1;
                    if (ab && Lb >= 0 && Lb <= p.max_len && Lb + 1 <= p.capacity)
                        len[bb] = Lb + 1;
                }
                if (lane == 0)
                    *p.append_counter = 0;
            }
        }
    } else if (warp == 0) {
        // =============================== TMA producer ===================================
        // The whole warp runs the loop; each lane issues at most one TMA box per tile (a
        // 64-column half of K or V for one page / block of rows), and lane 0 publishes the
        // tile with a single arrive.expect_tx of the warp's summed bytes.
        int issued = 0;
        if (n_tiles > 0) {
            const uint64_t pol = policy_evict_first();
            long long g = g0;
            int layer, b, kvh, t;
            first_tile(layer, b, kvh, t);
            auto ntiles_of = [&](int bb) { return c.nt[bb]; };
            int seg = -1;
            int seg_len = 0, seg_rows_c = 0, seg_ws = 0;
            // Sparse step: per-segment values loaded ahead of use, so the producer does not
            // wait on global memory at the tile that needs them. Lanes 0 and 1 hold the packed
            // row count and selection count of the current (cur_meta) and the next (nxt_meta)
            // segment, the next loaded when the current one starts; lane j < n_wbox holds the
            // page of window box j of the current segment (paged cache, up to 32 boxes).
            int cur_meta = 0, nxt_meta = 0, wpage = 0, seg_jn = 0;
            const bool wpage_pf = !DENSE && p.page_size != 0 && p.n_wbox <= 32;
            const int my_q = lane >> 2, my_op = lane & 3;  // page / block and (K|V, half)
            // paged dense tiles: this lane's page id, loaded one tile ahead
            const bool paged_dense = DENSE && p.page_size != 0;
            int my_page = 0;
            auto load_page = [&](int bb, int tt) {
                my_page = (tt * kTile + 16 * my_q < c.len[bb])
                              ? __ldg(p.page_table + bb * p.max_pages + tt * 8 + my_q)
                              : 0;
            };
            if (paged_dense)
                load_page(b, t);
            // Fused append: unit uu's new K and V rows go to cache position pos, 16 bytes per
            // lane (lanes 0-15 K, 16-31 V); each lane then fences its write against the async
            // proxy and the warp synchronises, so every later TMA box of this warp that covers
            // the row reads the new data. Issued right after the segment's first TMA (or before
            // it, when the first tile itself holds the row), well ahead of the box that reads it.
            auto append_row = [&](int uu, int ll, int bb, int kk, int pos) {
                long long row;
                bool good = true;
                if (p.page_size == 0) {
                    row = static_cast<long long>(uu) * p.capacity + pos;
                } else {
                    // the page of window box seg_jn from the segment's prefetch (all lanes take
                    // part in the shuffle), or, for a row outside the window (a sequence no
                    // longer than its sinks) and in the dense step, a direct lookup
                    int page = wpage_pf ? __shfl_sync(0xffffffffu, wpage, max(0, min(seg_jn, 31))) : 0;
                    if (!wpage_pf || seg_jn < 0 || seg_jn >= min(p.n_wbox, 32))
                        page = __ldg(p.page_table + bb * p.max_pages + (pos >> 4));
                    good = page >= 0 && page < p.n_pages;
                    if (!good && lane == 0)
                        raise_error(p.err, 0x1u);  // SFI_DEVERR_PAGE_RANGE
                    row = ((static_cast<long long>(ll) * p.n_pages + page) * Hkv + kk) * 16 + (pos & 15);
                }
                if (good) {
                    const int kvsel = lane >> 4, chunk = lane & 15;
                    const uint4 x = static_cast<const uint4 *>(kvsel ? p.v_new : p.k_new)
                        [static_cast<size_t>(uu) * 16 + chunk];
                    static_cast<uint4 *>(kvsel ? p.v_cache : p.k_cache)[row * 16 + chunk] = x;
                    fence_proxy_async_global();
                }
                __syncwarp();
            };
            int app_tile = -1;       // tile of the current segment that holds the new row
            bool appended = false;
            bool ok = true;
            bool pre_issued = false;  // the first tile's boxes were requested ahead (below)
            for (int i = 0; i < n_tiles; ++i, ++g) {
                if (i > 0 && ++t == ntiles_of(b)) {
                    t = 0;
                    if (++kvh == Hkv) {
                        kvh = 0;
                        do {
                            if (++b == B) {
                                b = 0;
                                ++layer;
                            }
                        } while (ntiles_of(b) == 0);
                    }
                }
                const int s = i % kStages;
                if (lane == 0)
                    ok = mbar_wait(&c.emptyK[s], ((i / kStages) & 1) ^ 1, &c.abort);
                const int u = (layer * B + b) * Hkv + kvh;
                const bool first = (i == 0) || (t == 0);
                const bool last = (i == n_tiles - 1) || (t == ntiles_of(b) - 1);
                // Sparse step: the range's first tile, when it holds packed rows only, is
                // requested at once with the query, every box of it, before the unit's packed
                // count and window start (two dependent global round trips) are known; its row
                // mask is published once they are (rows past the packed count are masked, and
                // their V rows zeroed, as in any tile).
                if (!DENSE && i == 0 && (t + 1) * kTile <= 64 * p.n_cbox &&
                    __shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
                    const int h2 = lane >> 4, j16 = lane & 15, kv0 = j16 >> 1, half0 = j16 & 1;
                    const int y0 = u * p.comp_cap + t * kTile + 64 * h2;
                    uint8_t *dst0 = smem + kv0 * 2 * kChunkBytes + half0 * kChunkBytes + 64 * h2 * 128;
                    if (lane == 0) {
                        TileMeta &mt = c.meta[0];
                        mt.unit = u;
                        mt.tile = t;
                        mt.flags = kFlagFirst | (last ? kFlagLast : 0);
                        mbar_arrive_expect_tx(&c.fullK[0], 2u * 2u * 64u * 128u + 2u * G * 128u +
                                                               ((p.test_stall && blockIdx.x == 0) ? 16u : 0u));
                    }
                    __syncwarp();
                    if (lane < 2)
                        tma_load_2d(smem + kQOff + lane * kOpChunk, &tm_q, &c.fullK[0], 64 * lane, u * G);
                    if (j16 < 2)
                        tma_load_2d(dst0, &tm_kc, &c.fullK[0], 64 * half0, y0);
                    issued = 1;
                    pre_issued = true;
                    bool okv = true;
                    if (lane == 0)
                        okv = mbar_wait(&c.emptyV[0], 1, &c.abort);
                    if (!__shfl_sync(0xffffffffu, okv ? 1 : 0, 0)) {
                        if (lane == 0) {   // no V requested: complete its phase for the drain
                            mbar_arrive(&c.fullV[0]);
                            fail(c, p.err);
                        }
                        break;
                    }
                    if (lane == 0)
                        mbar_arrive_expect_tx(&c.fullV[0], 2u * 2u * 64u * 128u);
                    __syncwarp();
                    if (j16 >= 2 && j16 < 4)
                        tma_load_2d(dst0, &tm_vc, &c.fullV[0], 64 * half0, y0);
                }
                const bool pre = pre_issued && i == 0;
                if (first) {
                    ++seg;
                    if (lane == 0 && ok && seg >= 2)
                        ok = mbar_wait(&c.q_free[seg & 1], ((seg >> 1) - 1) & 1, &c.abort);
                    seg_len = c.len[b];
                    if (!DENSE) {
                        int rows_c, sel;
                        {
                            cur_meta = seg == 0 ? (lane == 0 ? __ldg(p.comp_rows + u)
                                                   : lane == 1 ? __ldg(p.sel_cnt + u) : 0)
                                                : nxt_meta;
                            // the next segment of the range, if any: its counts, loaded now
                            if (i + (ntiles_of(b) - t) < n_tiles) {
                                int nl = layer, nb = b, nk = kvh;
                                if (++nk == Hkv) {
                                    nk = 0;
                                    do {
                                        if (++nb == B) {
                                            nb = 0;
                                            ++nl;
                                        }
                                    } while (ntiles_of(nb) == 0);
                                }
                                const int un = (nl * B + nb) * Hkv + nk;
                                nxt_meta = lane == 0 ? __ldg(p.comp_rows + un)
                                                     : lane == 1 ? __ldg(p.sel_cnt + un) : 0;
                            }
                            rows_c = __shfl_sync(0xffffffffu, cur_meta, 0);
                            sel = __shfl_sync(0xffffffffu, cur_meta, 1);
                        }
                        rows_c = max(0, min(rows_c, p.comp_cap));
                        const int n_s = max(0, rows_c - max(0, sel));
                        seg_rows_c = rows_c;
                        seg_ws = max(n_s, seg_len - p.n_window);
                        if (wpage_pf) {
                            const int lp = (seg_ws >> 4) + lane;
                            wpage = (lane < p.n_wbox && lp * 16 < seg_len)
                                        ? __ldg(p.page_table + b * p.max_pages + lp) : 0;
                        }
                    }
                    if (fused) {
                        const int Ln = seg_len - 1;  // position of the new row
                        int t_new;
                        if (DENSE) {
                            t_new = Ln / kTile;  // the tile of the unit's positions that holds it
                        } else {
                            const int jn = p.page_size == 0 ? ((Ln - seg_ws) >> 4)
                                                            : ((Ln >> 4) - (seg_ws >> 4));
                            seg_jn = jn;
                            t_new = (64 * p.n_cbox + 16 * jn) / kTile;
                        }
                        const int t_end = min(ntiles_of(b) - 1, t + (n_tiles - 1 - i));
                        app_tile = (seg_len >= 1 && t_new >= t && t_new <= t_end) ? t_new : -1;
                        appended = false;
                    }
                }
                if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
                    if (lane == 0)
                        fail(c, p.err);
                    break;
                }
                const int L = seg_len;
                // page of this lane's window box, from the segment's prefetch (all lanes take
                // part in the shuffle; lanes without a window box ignore the value)
                int wpg = 0;
                if (wpage_pf && (t + 1) * kTile > 64 * p.n_cbox) {   // a tile with window boxes
                    const int jl = (t * kTile + 64 * (lane >> 4) + 16 * ((lane & 15) >> 2) -
                                    64 * p.n_cbox) >> 4;
                    wpg = __shfl_sync(0xffffffffu, wpage, jl & 31);
                }
                // ---- this lane's box ----------------------------------------------------
                const CUtensorMap *map = nullptr;
                int y = 0, row0 = 0, rows = 0, kv = 0, half = 0;
                uint32_t valid[4] = {0u, 0u, 0u, 0u};
                if (DENSE) {
                    const int pos0 = t * kTile;
                    const int nvalid = min(kTile, L - pos0);
                    if (p.page_size == 0) {
                        if (lane == 0)
                            mask_rows(valid, 0, nvalid);
                        if (lane < 4) {
                            kv = lane >> 1;
                            half = lane & 1;
                            map = kv ? &tm_v : &tm_k;
                            y = u * p.capacity + pos0;
                            rows = kTile;
                        }
                    } else if (16 * my_q < nvalid) {
                        if (my_page < 0 || my_page >= p.n_pages) {
                            if (my_op == 0)
                                raise_error(p.err, 0x1u);  // rows of this page stay invalid
                        } else {
                            kv = my_op >> 1;
                            half = my_op & 1;
                            map = kv ? &tm_v : &tm_k;
                            y = ((layer * p.n_pages + my_page) * Hkv + kvh) * 16;
                            row0 = 16 * my_q;
                            rows = 16;
                            if (my_op == 0)
                                mask_rows(valid, row0, min(row0 + 16, nvalid));
                        }
                    }
                } else {
                    const int h2 = lane >> 4, j16 = lane & 15;
                    const int R = t * kTile + 64 * h2;
                    if (R < 64 * p.n_cbox) {
                        const int k = R >> 6;
                        const int vr = max(0, min(64, seg_rows_c - 64 * k));
                        if (vr > 0 && j16 < 4) {
                            kv = j16 >> 1;
                            half = j16 & 1;
                            map = kv ? &tm_vc : &tm_kc;
                            y = u * p.comp_cap + 64 * k;
                            row0 = 64 * h2;
                            rows = 64;
                            if (j16 == 0)
                                mask_rows(valid, row0, row0 + vr);
                        }
                    } else {
                        const int q = j16 >> 2;
                        const int j = (R + 16 * q - 64 * p.n_cbox) >> 4;
                        const int rr0 = 64 * h2 + 16 * q;
                        if (j < p.n_wbox && p.page_size == 0) {
                            const int p0 = seg_ws + 16 * j;
                            const int vr = max(0, min(16, L - p0));
                            if (vr > 0) {
                                kv = my_op >> 1;
                                half = my_op & 1;
                                map = kv ? &tm_v : &tm_k;
                                y = u * p.capacity + p0;
                                row0 = rr0;
                                rows = 16;
                                if (my_op == 0)
                                    mask_rows(valid, rr0, rr0 + vr);
                            }
                        } else if (j < p.n_wbox) {
                            const int lp = (seg_ws >> 4) + j;
                            const int r0 = max(seg_ws - lp * 16, 0);
                            const int r1 = min(L - lp * 16, 16);
                            if (r1 > r0) {
                                const int page = wpage_pf ? wpg
                                                          : __ldg(p.page_table + b * p.max_pages + lp);
                                if (page < 0 || page >= p.n_pages) {
                                    if (my_op == 0)
                                        raise_error(p.err, 0x1u);
                                } else {
                                    kv = my_op >> 1;
                                    half = my_op & 1;
                                    map = kv ? &tm_v : &tm_k;
                                    y = ((layer * p.n_pages + page) * Hkv + kvh) * 16;
                                    row0 = rr0;
                                    rows = 16;
                                    if (my_op == 0)
                                        mask_rows(valid, rr0 + r0, rr0 + r1);
                                }
                            }
                        }
                    }
                }
                if (fused && app_tile == t && !appended) {  // this tile holds the new row
                    append_row(u, layer, b, kvh, L - 1);
                    appended = true;
                }
                // ---- publish the tile, then issue ---------------------------------------
                uint32_t vw[4];
#pragma unroll
                for (int w = 0; w < 4; ++w)
                    vw[w] = __reduce_or_sync(0xffffffffu, valid[w]);
                // test hook: CTA 0's first tile expects 16 bytes that never come, so the waits
                // on it run out (see sfi_test_inject_stall)
                const uint32_t bytes_k =
                    __reduce_add_sync(0xffffffffu, kv == 0 ? static_cast<uint32_t>(rows) * 128u : 0u) +
                    (first ? 2u * G * 128u : 0u) +
                    ((p.test_stall && blockIdx.x == 0 && i == 0) ? 16u : 0u);
                const uint32_t bytes_v =
                    __reduce_add_sync(0xffffffffu, kv == 1 ? static_cast<uint32_t>(rows) * 128u : 0u);
                if (lane == 0) {
                    TileMeta &mt = c.meta[i % kMetaRing];
                    if (!pre) {
                        mt.unit = u;
                        mt.tile = t;
                        mt.flags = (first ? kFlagFirst : 0) | (last ? kFlagLast : 0);
                    }
#pragma unroll
                    for (int w = 0; w < 4; ++w)
                        mt.valid[w] = vw[w];
                    mbar_arrive(&c.meta_full[i % kMetaRing]);  // releases the metadata
                    if (!pre)
                        mbar_arrive_expect_tx(&c.fullK[s], bytes_k);  // (and for the MMA's flags)
                }
                __syncwarp();
                if (pre) {
                    // requested ahead; only the append may remain
                    if (fused && app_tile >= 0 && !appended) {
                        append_row(u, layer, b, kvh, L - 1);
                        appended = true;
                    }
                    continue;
                }
                if (first && lane < 2) {
                    uint8_t *qb = smem + kQOff + (seg & 1) * kOpBytes;
                    tma_load_2d(qb + lane * kOpChunk, &tm_q, &c.fullK[s], 64 * lane, u * G);
                }
                uint8_t *dst = smem + s * kStageBytes + kv * 2 * kChunkBytes + half * kChunkBytes +
                               row0 * 128;
                // K half now; the V half once the P.V MMA of this stage's previous tile is done
                if (rows > 0 && kv == 0) {
                    if (DENSE)  // streamed once per slow step: do not displace reusable lines
                        tma_load_2d_hint(dst, map, &c.fullK[s], 64 * half, y, pol);
                    else
                        tma_load_2d(dst, map, &c.fullK[s], 64 * half, y);
                }
                bool okv = true;
                if (lane == 0)
                    okv = mbar_wait(&c.emptyV[s], ((i / kStages) & 1) ^ 1, &c.abort);
                if (!__shfl_sync(0xffffffffu, okv ? 1 : 0, 0)) {
                    if (lane == 0) {   // no V requested: complete its phase for the drain
                        mbar_arrive(&c.fullV[s]);
                        fail(c, p.err);
                    }
                    ++issued;
                    break;
                }
                if (lane == 0)
                    mbar_arrive_expect_tx(&c.fullV[s], bytes_v);
                __syncwarp();
                if (rows > 0 && kv == 1) {
                    if (DENSE)
                        tma_load_2d_hint(dst, map, &c.fullV[s], 64 * half, y, pol);
                    else
                        tma_load_2d(dst, map, &c.fullV[s], 64 * half, y);
                }
                if (fused && app_tile >= 0 && !appended) {  // a later tile holds it
                    append_row(u, layer, b, kvh, L - 1);
                    appended = true;
                }
                ++issued;
                if (paged_dense && i + 1 < n_tiles) {
                    int nb = b, nt2 = t + 1;
                    if (nt2 == c.nt[b]) {
                        nt2 = 0;
                        if (kvh + 1 == Hkv) {
                            do {
                                if (++nb == B)
                                    nb = 0;
                            } while (c.nt[nb] == 0);
                        }
                    }
                    load_page(nb, nt2);
                }
            }
        }
        // Never leave a copy in flight into shared memory we are about to give up.
        if (lane == 0)
            for (int j = max(0, issued - kStages); j < issued; ++j) {
                mbar_wait(&c.fullK[j % kStages], (j / kStages) & 1, nullptr);
                mbar_wait(&c.fullV[j % kStages], (j / kStages) & 1, nullptr);
            }
        // Fused append: this CTA has read seq_len (set-up); the last CTA of the grid to get
        // here advances the length of every sequence whose new row was appended.
        if (fused) {
            int is_last = 0;
            if (lane == 0)
                is_last = atomic_add_acq_rel_gpu(p.append_counter, 1) == static_cast<int>(gridDim.x) - 1;
            if (__shfl_sync(0xffffffffu, is_last, 0)) {
                int32_t *len = const_cast<int32_t *>(p.seq_len);
                for (int bb = lane; bb < B; bb += 32) {
                    const int L0 = len[bb];
                    const int act = p.active ? p.active[bb] : 1;
                    if (act && L0 >= 0 && L0 <= p.max_len && L0 + 1 <= p.capacity)
                        len[bb] = L0 + 1;
                }
                if (lane == 0)
                    *p.append_counter = 0;
            }
        }
    } else if (warp == 1) {
        // ================================ MMA issuer =====================================
        // One thread issues, in tile order, S(i) = K_i Q^T once tile i has landed and its S
        // buffer is free, and O(i) = V_i^T P_i^T once the softmax has written P_i: whichever
        // is ready first, so a slow softmax on one tile does not hold back the next S.
        if (lane == 0 && n_tiles > 0) {
            constexpr uint32_t idesc_s = idesc_bf16(kTile, kOpRows, false, false);
            constexpr uint32_t idesc_o = idesc_bf16(kTile, kOpRows, true, false);
            int seg = -1, ns = 0, np = 0;
            bool ok = true;
            uint32_t idle = 0;
            uint64_t idle_t0 = 0;
            while (np < n_tiles) {
                bool prog = false;
                if (ns < n_tiles) {
                    const int s = ns % kStages, bb = ns & 1, use = ns >> 1;
                    // (clustered: the query has its own barrier, awaited before the first S)
                    if (mbar_test_wait(&c.fullK[s], (ns / kStages) & 1) &&
                        mbar_test_wait(&c.s_free[bb], (use & 1) ^ 1) &&
                        (!clustered || ns > 0 || mbar_test_wait(&c.q_full, 0))) {
                        // clustered: the row masks may still be in flight; the flags are static
                        const int flags = clustered ? ((ns == 0 ? kFlagFirst : 0) |
                                                       (ns == n_tiles - 1 ? kFlagLast : 0))
                                                    : c.meta[ns % kMetaRing].flags;
                        if (flags & kFlagFirst)
                            ++seg;
                        tc_fence_after();
                        const uint32_t ka = smem_u32(smem + s * kStageBytes);
                        const uint32_t qa = smem_u32(smem + kQOff + (seg & 1) * kOpBytes);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint64_t a = smem_desc_sw128(ka + (kk >> 2) * kChunkBytes + (kk & 3) * 32, 16, 1024);
                            const uint64_t bd = smem_desc_sw128(qa + (kk >> 2) * kOpChunk + (kk & 3) * 32, 16, 1024);
                            umma_bf16(tmem + bb * 16, a, bd, idesc_s, kk > 0 ? 1u : 0u);
                        }
                        umma_commit(&c.s_full[bb]);
                        umma_commit(&c.emptyK[s]);   // the K half is free once S is done
                        if (flags & kFlagLast)
                            umma_commit(&c.q_free[seg & 1]);
                        ++ns;
                        prog = true;
                    }
                }
                if (np < ns) {
                    const int s = np % kStages, bb = np & 1, use = np >> 1;
                    if (mbar_test_wait(&c.p_full[bb], use & 1) &&
                        mbar_test_wait(&c.o_free[bb], (use & 1) ^ 1) &&
                        mbar_test_wait(&c.fullV[s], (np / kStages) & 1)) {
                        tc_fence_after();
                        const uint32_t va = smem_u32(smem + s * kStageBytes + 2 * kChunkBytes);
                        const uint32_t pa = smem_u32(smem + kPOff + bb * kOpBytes);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint64_t a = smem_desc_sw128(va + kk * 2048, kChunkBytes, 1024);
                            const uint64_t bd = smem_desc_sw128(pa + (kk >> 2) * kOpChunk + (kk & 3) * 32, 16, 1024);
                            umma_bf16(tmem + 32 + bb * 16, a, bd, idesc_o, kk > 0 ? 1u : 0u);
                        }
                        umma_commit(&c.o_full[bb]);
                        umma_commit(&c.emptyV[s]);
                        ++np;
                        prog = true;
                    }
                }
                if (prog) {
                    idle = 0;
                    continue;
                }
                // nothing ready: poll again (the softmax warps leave most issue slots free);
                // give up after kWaitTimeoutNs without progress, or as soon as another role
                // has given up
                if ((++idle & 63u) == 0u) {
                    if (c.abort) {
                        ok = false;
                        break;
                    }
                    const uint64_t now = global_timer_ns();
                    if (idle == 64u)
                        idle_t0 = now;
                    else if (now - idle_t0 > kWaitTimeoutNs) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok)
                fail(c, p.err);
            // All MMAs of this thread are complete once `drain` fires.
            umma_commit(&c.drain);
            mbar_wait(&c.drain, 0, nullptr);
        }
    } else {
        // ========================= softmax / epilogue warps ============================
        const int wq = warp & 3;              // TMEM lane quarter this warp may access
        const int row = wq * 32 + lane;       // S^T row (tile position) / O^T row (dim)
        const int gw = warp - 2;              // index within the softmax group
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        uint32_t gphase = 0;
        float m_run[G], le[G], acc[G];
        // the tile waiting for its O^T accumulation
        float a_alpha[G], a_m[G], a_le[G];
        // clustered: this CTA's (max, sum) of its slice, with acc[] its unnormalised output
        float fin_m[G], fin_le[G];
        int a_flags = 0, a_unit = 0;
        bool ok = true;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            m_run[h] = -INFINITY;
            le[h] = acc[h] = 0.f;
            fin_m[h] = -INFINITY;
            fin_le[h] = 0.f;
        }

        auto finalize = [&](int u, const float (&fm)[G], const float (&fle)[G]) -> bool {
            const int kvh = u % Hkv, b = (u / Hkv) % B, layer = u / (Hkv * B);
            // sparse: an active sequence found with an invalid or empty length gives no output
            // (every CTA of the unit sees the same length, so none takes part in its merge)
            if (!DENSE && c.len[b] <= 0)
                return true;
            const long long su = layer * c.TL + c.pre[b] + static_cast<long long>(kvh) * c.nt[b];
            const long long eu = su + c.nt[b];
            const long long P = c.P, T = c.T;
            // the CTAs whose stream-K ranges meet [su, eu)
            const int cf = static_cast<int>(((su + 1) * P - 1) / T);
            const int cl = static_cast<int>((eu * P - 1) / T);
            float o[G];
            if (cf == cl) {
#pragma unroll
                for (int h = 0; h < G; ++h)
                    o[h] = fle[h] > 0.f ? acc[h] / fle[h] : 0.f;
                store_out<G>(p, u, row, o);
                if (DENSE && row < G)
                    p.stats[u * G + row] = make_float2(pick<G>(fm, row), pick<G>(fle, row));
                return true;
            }
            const int slot = (su <= g0) ? 0 : 1;
            float *part = p.partials + (2 * static_cast<size_t>(blockIdx.x) + slot) * kPartialFloats(G);
            // dim-major [128][G]: one 16-byte store (and load in the merge) per dim for G >= 4
            if constexpr (G >= 4) {
#pragma unroll
                for (int h = 0; h < G; h += 4)
                    *reinterpret_cast<float4 *>(part + row * G + h) =
                        make_float4(acc[h], acc[h + 1], acc[h + 2], acc[h + 3]);
            } else {
#pragma unroll
                for (int h = 0; h < G; ++h)
                    part[row * G + h] = acc[h];
            }
            if (row < G) {
                part[G * kHeadDim + row] = pick<G>(fm, row);
                part[G * kHeadDim + G + row] = pick<G>(fle, row);
            }
            // Every thread's partial writes happen before thread 0's release fence (group
            // barrier), which publishes them before the ticket; the last contributor's
            // acquire fence and the second barrier make all partials visible to its threads.
            if (!group_sync(c, gphase, lane))
                return false;
            if (row == 0) {
                fence_acq_rel_gpu();
                const int tk = atomicAdd(&p.tickets[u], 1);
                const int is_last = (tk == cl - cf) ? 1 : 0;
                if (is_last) {
                    p.tickets[u] = 0;
                    fence_acq_rel_gpu();
                }
                c.last_flag = is_last;
            }
            if (!group_sync(c, gphase, lane))
                return false;
            if (!c.last_flag)
                return true;
            // Merge over the contributors in CTA order (this CTA's own partial from registers
            // at its place), so the rounding does not depend on which contributor arrived
            // last, in chunks of up to 32 contributors. Lane k of every softmax warp loads
            // contributor c0 + k's maxima and weight sums; a warp max gives the chunk's
            // maximum M, and each contributor's weight 2^(m_k - M) is computed once, in its
            // lane, rather than by every thread. Each thread then sums its dim of the
            // contributors' outputs with those weights (taken by shuffle), kSB contributors'
            // loads at a time, the first kSB issued together with the maxima. (A per-thread
            // online merge spent ~2.9 us per 8 contributors: a one-sequence launch, whose units
            // are split over ~20 CTAs, ended ~9 us after its last tile.)
            constexpr int kSB = G <= 4 ? 8 : 4;
            float M[G], Le[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                M[h] = -INFINITY;
                Le[h] = 0.f;
                o[h] = 0.f;
            }
            // u may be the last segment of cf's range (slot 1)
            const bool cf_tail = static_cast<long long>(cf) * T / P < su;
            auto part_of = [&](int cc) -> const float * {
                const int sl = (cc == cf && cf_tail) ? 1 : 0;
                return p.partials + (2 * static_cast<size_t>(cc) + sl) * kPartialFloats(G);
            };
            for (int c0 = cf; c0 <= cl; c0 += 32) {
                const int nk = min(32, cl - c0 + 1);
                // this dim of contributors c0 + k0 .. c0 + k0 + kSB - 1
                float a[kSB][G];
                auto load_out = [&](int k0) {
#pragma unroll
                    for (int j = 0; j < kSB; ++j) {
                        const int cc = c0 + k0 + j;
                        if (k0 + j < nk && cc != static_cast<int>(blockIdx.x)) {
                            const float *pc = part_of(cc);
                            if constexpr (G >= 4) {
#pragma unroll
                                for (int h = 0; h < G; h += 4) {
                                    const float4 x = __ldcg(reinterpret_cast<const float4 *>(pc + row * G + h));
                                    a[j][h] = x.x;
                                    a[j][h + 1] = x.y;
                                    a[j][h + 2] = x.z;
                                    a[j][h + 3] = x.w;
                                }
                            } else {
#pragma unroll
                                for (int h = 0; h < G; ++h)
                                    a[j][h] = __ldcg(pc + row * G + h);
                            }
                        } else {
#pragma unroll
                            for (int h = 0; h < G; ++h)
                                a[j][h] = (k0 + j < nk) ? acc[h] : 0.f;
                        }
                    }
                };
                load_out(0);
                // lane k: maxima and weight sums of contributor c0 + k
                float mk[G], lk[G];
                {
                    const int ck = c0 + lane;
                    if (lane < nk && ck != static_cast<int>(blockIdx.x)) {
                        const float *pc = part_of(ck);
#pragma unroll
                        for (int h = 0; h < G; ++h) {
                            mk[h] = __ldcg(pc + G * kHeadDim + h);
                            lk[h] = __ldcg(pc + G * kHeadDim + G + h);
                        }
                    } else {
#pragma unroll
                        for (int h = 0; h < G; ++h) {
                            mk[h] = lane < nk ? fm[h] : -INFINITY;
                            lk[h] = lane < nk ? fle[h] : 0.f;
                        }
                    }
                }
                float wk[G];
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float mn = fmaxf(M[h], warp_max(mk[h]));
                    const float mb = (mn == -INFINITY) ? 0.f : mn;
                    const float sc = ex2_approx(M[h] - mb);     // 0 while nothing is merged
                    wk[h] = ex2_approx(mk[h] - mb);              // 0 for an empty contributor
                    o[h] *= sc;
                    Le[h] = fmaf(Le[h], sc, warp_sum(wk[h] * lk[h]));
                    M[h] = mn;
                }
#pragma unroll 1
                for (int k0 = 0; k0 < nk; k0 += kSB) {
                    if (k0 > 0)
                        load_out(k0);
#pragma unroll
                    for (int j = 0; j < kSB; ++j) {
#pragma unroll
                        for (int h = 0; h < G; ++h) {
                            const float w = __shfl_sync(0xffffffffu, wk[h], (k0 + j) & 31);
                            if (k0 + j < nk)
                                o[h] = fmaf(w, a[j][h], o[h]);
                        }
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < G; ++h)
                o[h] = Le[h] > 0.f ? o[h] / Le[h] : 0.f;
            store_out<G>(p, u, row, o);
            if (DENSE && row < G)
                p.stats[u * G + row] = make_float2(pick<G>(M, row), pick<G>(Le, row));
            return true;
        };

        auto correct = [&](int j) -> bool {
            const int bb = j & 1, use = j >> 1;
            if (!mbar_wait(&c.o_full[bb], use & 1, &c.abort))
                return false;
            float ov2[2 * G], ov[G];
            tmem_load<2 * G>(t_lane + 32 + bb * 16, ov2);
#pragma unroll
            for (int h = 0; h < G; ++h)
                ov[h] = ov2[h] + ov2[G + h];
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&c.o_free[bb]);
#pragma unroll
            for (int h = 0; h < G; ++h)
                acc[h] = (a_flags & kFlagFirst) ? ov[h] : fmaf(acc[h], a_alpha[h], ov[h]);
            if (a_flags & kFlagLast) {
                if (clustered) {  // merged across the cluster after the loop
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        fin_m[h] = a_m[h];
                        fin_le[h] = a_le[h];
                    }
                    return true;
                }
                if (!finalize(a_unit, a_m, a_le))
                    return false;
#pragma unroll
                for (int h = 0; h < G; ++h)
                    acc[h] = 0.f;
            }
            return true;
        };

        for (int i = 0; i < n_tiles && ok; ++i) {
            const int s = i % kStages, bb = i & 1, use = i >> 1;
            // the tile's scores, then its metadata (row mask), published on the ring's own
            // barrier (for a clustered step possibly after the data)
            if (!mbar_wait(&c.s_full[bb], use & 1, &c.abort) ||
                !mbar_wait(&c.meta_full[i % kMetaRing], (i / kMetaRing) & 1, &c.abort)) {
                ok = false;
                break;
            }
            const TileMeta &mt = c.meta[i % kMetaRing];
            const int u = mt.unit;
            const int tile = mt.tile;
            const int flags = mt.flags;
            const bool valid = (mt.valid[row >> 5] >> (row & 31)) & 1u;
            if (flags & kFlagFirst) {
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    m_run[h] = -INFINITY;
                    le[h] = 0.f;
                }
            }
            float sv[G];
            tmem_load<G>(t_lane + bb * 16, sv);
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&c.s_free[bb]);
            float z[G];
#pragma unroll
            for (int h = 0; h < G; ++h)
                z[h] = valid ? sv[h] * p.scale_log2 : -INFINITY;
            if (DENSE && p.zbuf != nullptr && valid) {
                float *zp = p.zbuf + (static_cast<size_t>(u) * p.capacity + tile * kTile + row) * G;
                if constexpr (G == 4) {
                    *reinterpret_cast<float4 *>(zp) = make_float4(z[0], z[1], z[2], z[3]);
                } else {
#pragma unroll
                    for (int h = 0; h < G; ++h)
                        zp[h] = z[h];
                }
            }
            // tile max over the 128 positions, per head
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float wm = warp_max(z[h]);
                if (lane == 0)
                    c.red_max[i & 1][gw][h] = wm;
            }
            if (!group_sync(c, gphase, lane)) {
                ok = false;
                break;
            }
            float alpha[G];
            uint8_t *pb = smem + kPOff + bb * kOpBytes;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float tm = fmaxf(fmaxf(c.red_max[i & 1][0][h], c.red_max[i & 1][1][h]),
                                       fmaxf(c.red_max[i & 1][2][h], c.red_max[i & 1][3][h]));
                const float mn = fmaxf(m_run[h], tm);
                const float mb = (mn == -INFINITY) ? 0.f : mn;
                alpha[h] = ex2_approx(m_run[h] - mb);
                const float pe = valid ? ex2_approx(z[h] - mb) : 0.f;
                const __nv_bfloat16 phi = __float2bfloat16_rn(pe);
                const __nv_bfloat16 plo = __float2bfloat16_rn(pe - __bfloat162float(phi));
                // phi + plo equals pe to about 2^-17, so the fp32 sum also normalises the O^T
                // the MMAs accumulate from the two parts
                le[h] = fmaf(le[h], alpha[h], pe);
                m_run[h] = mn;
                // P^T[h][row] and P^T[G + h][row], K-major, 128-byte swizzle
                const int base = (row >> 6) * kOpChunk + (row & 7) * 2;
                const int sw = (row & 63) >> 3;
                *reinterpret_cast<__nv_bfloat16 *>(pb + base + h * 128 + ((sw ^ h) << 4)) = phi;
                *reinterpret_cast<__nv_bfloat16 *>(pb + base + (G + h) * 128 +
                                                   ((sw ^ ((G + h) & 7)) << 4)) = plo;
            }
            bool vok = true;
            if (!valid) {
                // keep P = 0 rows from meeting stale (possibly non-finite) V data, once the
                // tile's V half has landed (it may follow the K half)
                vok = mbar_wait(&c.fullV[s], (i / kStages) & 1, &c.abort);
                uint8_t *vrow = smem + s * kStageBytes + 2 * kChunkBytes + row * 128;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    reinterpret_cast<uint4 *>(vrow)[k] = make_uint4(0u, 0u, 0u, 0u);
                    reinterpret_cast<uint4 *>(vrow + kChunkBytes)[k] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            if (!__all_sync(0xffffffffu, vok)) {
                ok = false;
                break;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&c.p_full[bb]);
            float fm[G], fle[G];
            if (flags & kFlagLast) {
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float s1 = warp_sum(le[h]);
                    if (lane == 0)
                        c.red_sum[gw][h] = s1;
                }
                if (!group_sync(c, gphase, lane)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    fm[h] = m_run[h];
                    fle[h] = c.red_sum[0][h] + c.red_sum[1][h] + c.red_sum[2][h] + c.red_sum[3][h];
                }
            }
            if (i > 0 && !correct(i - 1)) {
                ok = false;
                break;
            }
            // this tile now waits for its accumulation
#pragma unroll
            for (int h = 0; h < G; ++h) {
                a_alpha[h] = alpha[h];
                if (flags & kFlagLast) {
                    a_m[h] = fm[h];
                    a_le[h] = fle[h];
                }
            }
            a_flags = flags;
            a_unit = u;
            (void)tile;
        }
        if (ok && n_tiles > 0 && !correct(n_tiles - 1))
            ok = false;
        // clustered: the unit's liveness is published by the producer with unit_meta (it
        // arrives there before its first wait, so this completes unless it never started)
        bool meta_ok = true;
        if (clustered && !(meta_ok = mbar_wait(&c.unit_meta, 0, &c.abort)))
            ok = false;
        if (clustered && meta_ok && c.cl_live) {
            // ---- merge the cluster's partials through distributed shared memory ----------
            // CTA r owns dims [r 128/C, (r+1) 128/C). Every CTA pushes, with asynchronous
            // remote stores that count their bytes on the owner's cl_ready, its (max, sum)
            // and its unnormalised outputs of each owner's dims into that owner's receive area
            // (the second Q buffer: a clustered CTA has one segment and uses only the first);
            // each owner expects all C sources' bytes on its own barrier. An owner whose
            // barrier has completed merges from its own shared memory; after that no peer
            // touches it, so it may exit. Every CTA of a live cluster pushes even after a
            // failed wait, so no peer waits for it; outputs are written only when everything
            // succeeded.
            cluster_wait_acquire();            // the peers' barriers are initialised
            const int C = p.cluster;           // 2, 4 or 8 (group <= 4: see the host)
            const int nd = kHeadDim / C;       // dims per owner
            const int rank = static_cast<int>(blockIdx.x) % C;
            const int u = static_cast<int>(blockIdx.x) / C;
            float *recv = reinterpret_cast<float *>(smem + kQOff + kOpBytes);
            // receive layout: acc [src][nd][G], then stats [src][G][2] (max, sum)
            const int acc_floats = C * G * nd;
            if (row == 0)   // every byte the C sources push here
                mbar_arrive_expect_tx(&c.cl_ready, static_cast<uint32_t>(C * (nd * G + 2 * G) * 4));
            {
                const int owner = row / nd, j = row - owner * nd;
                const uint32_t rb = map_to_rank(&c.cl_ready, static_cast<uint32_t>(owner));
                const uint32_t base = map_to_rank(recv, static_cast<uint32_t>(owner)) +
                                      4u * ((rank * nd + j) * G);
                if constexpr (G == 4) {
                    st_async_f32x4(base, acc[0], acc[1], acc[2], acc[3], rb);
                } else {
#pragma unroll
                    for (int h = 0; h < G; ++h)
                        st_async_f32(base + 4u * h, acc[h], rb);
                }
                if (row < C * G) {  // (max, sum) of head h to owner row / G
                    const int ow = row / G, h = row - ow * G;
                    const uint32_t b2 = map_to_rank(recv, static_cast<uint32_t>(ow)) +
                                        4u * (acc_floats + (rank * G + h) * 2);
                    st_async_f32x2(b2, pick<G>(fin_m, h), pick<G>(fin_le, h),
                                   map_to_rank(&c.cl_ready, static_cast<uint32_t>(ow)));
                }
            }
            bool good = ok;
            // A peer arrives within its own bounded waits even when it fails; this limit is
            // well above those, so no CTA leaves while a live peer may still push to it.
            good = mbar_wait_cluster(&c.cl_ready, 0, 8 * kWaitTimeoutNs) && good;
            if (good) {
                for (int o = row; o < nd * G; o += 4 * 32) {
                    const int h = o / nd, j = o - h * nd;
                    float M = -INFINITY;
                    for (int q = 0; q < C; ++q)
                        M = fmaxf(M, recv[acc_floats + (q * G + h) * 2]);
                    float Lsum = 0.f, O = 0.f;
                    for (int q = 0; q < C; ++q) {
                        const float mq = recv[acc_floats + (q * G + h) * 2];
                        const float w = (mq == -INFINITY) ? 0.f : exp2f(mq - M);
                        Lsum = fmaf(w, recv[acc_floats + (q * G + h) * 2 + 1], Lsum);
                        O = fmaf(w, recv[(q * nd + j) * G + h], O);
                    }
                    const float v = Lsum > 0.f ? O / Lsum : 0.f;
                    const size_t idx = (static_cast<size_t>(u) * G + h) * kHeadDim + rank * nd + j;
                    if (p.out_fp32)
                        static_cast<float *>(p.out)[idx] = v;
                    else
                        static_cast<__nv_bfloat16 *>(p.out)[idx] = __float2bfloat16_rn(v);
                }
            }
            if (!good)
                ok = false;
        }
        if (!ok)
            fail(c, p.err);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

constexpr int kEvPer = 4;   // positions per thread of the evidence kernel

// Evidence f_j = (1/G) sum_h exp2(z_hj - M_h) / L_h from the dense step's base-2 logits
// and merged statistics; one pass over [units][positions]. (The clustered Selector repeats
// this arithmetic, term for term, when it computes the evidence itself.)
template <int G>
__global__ void __launch_bounds__(256) evidence_kernel(const float *__restrict__ zbuf,
                                                       const float2 *__restrict__ stats,
                                                       float *__restrict__ f,
                                                       const int32_t *__restrict__ seq_len,
                                                       const uint8_t *__restrict__ active,
                                                       int batch, int n_kv_heads, int capacity,
                                                       int n_seq_active)
{
    pdl_trigger();
    pdl_wait();
    // (with n_seq_active > 0 the grid covers only the active sequences' units)
    const int u = launched_unit(static_cast<int>(blockIdx.y), n_seq_active, active, batch, n_kv_heads);
    if (u < 0)
        return;
    const int b = (u / n_kv_heads) % batch;
    if (active && !active[b])
        return;
    const int L = min(seq_len[b], capacity);
    float M[G], inv[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const float2 st = stats[u * G + h];
        M[h] = st.x;
        inv[h] = st.y > 0.f ? 1.f / st.y : 0.f;
    }
    const float rg = 1.f / static_cast<float>(G);
    const float *zu = zbuf + static_cast<size_t>(u) * capacity * G;
    float *fu = f + static_cast<size_t>(u) * capacity;
    // The grid covers the longest sequence with kEvPer positions per thread: all of a
    // thread's loads are issued before the first is used (one round trip, not kEvPer).
    const int stride = gridDim.x * blockDim.x;
    const int j0 = blockIdx.x * blockDim.x + threadIdx.x;
    float z[kEvPer][G];
#pragma unroll
    for (int r = 0; r < kEvPer; ++r) {
        const int j = j0 + r * stride;
        if (j < L) {
            if constexpr (G == 4) {
                const float4 v = __ldcs(reinterpret_cast<const float4 *>(zu) + j);
                z[r][0] = v.x; z[r][1] = v.y; z[r][2] = v.z; z[r][3] = v.w;
            } else {
#pragma unroll
                for (int h = 0; h < G; ++h)
                    z[r][h] = __ldcs(zu + static_cast<size_t>(j) * G + h);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kEvPer; ++r) {
        const int j = j0 + r * stride;
        if (j < L) {
            float acc = 0.f;
#pragma unroll
            for (int h = 0; h < G; ++h)
                acc = fmaf(exp2f(z[r][h] - M[h]), inv[h], acc);
            fu[j] = acc * rg;
        }
    }
    // (only a length above the launch's bound reaches here; the dense step flags it)
    for (int j = j0 + kEvPer * stride; j < L; j += stride) {
        float acc = 0.f;
#pragma unroll
        for (int h = 0; h < G; ++h)
            acc = fmaf(exp2f(__ldcs(zu + static_cast<size_t>(j) * G + h) - M[h]), inv[h], acc);
        fu[j] = acc * rg;
    }
}

template <int G, bool DENSE>
cudaError_t launch_attn_t(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                          const CUtensorMap &tm_kc, const CUtensorMap &tm_vc, const AttnParams &p,
                          int grid, cudaStream_t stream)
{
    const int cluster = (!DENSE && p.cluster > 1) ? p.cluster : 1;
    // dense: the instance with the fused append when p.k_new is set
    auto kern = cluster > 1 ? attn_kernel<G, false, true>
                            : (DENSE && p.k_new != nullptr) ? attn_kernel<G, DENSE, true>
                                                            : attn_kernel<G, DENSE, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess)
        return e;
    if (grid % cluster != 0)
        return cudaErrorInvalidValue;
    e = launch_pdl_cluster(kern, dim3(grid), dim3(kAttnThreads), kSmemBytes, cluster, stream, tm_k,
                           tm_v, tm_q, tm_kc, tm_vc, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Clusters of `cluster` sparse-kernel CTAs that can be resident at once on this device.
template <int G>
int max_active_clusters_t(int cluster)
{
    auto kern = attn_kernel<G, false, true>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cluster) * 64u);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
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

int max_active_clusters(int group, int cluster)
{
    switch (group) {
    case 1: return max_active_clusters_t<1>(cluster);
    case 2: return max_active_clusters_t<2>(cluster);
    case 4: return max_active_clusters_t<4>(cluster);
    case 8: return max_active_clusters_t<8>(cluster);
    default: return 0;
    }
}

constexpr int kMaxDevicesCached = 64;
std::mutex g_cluster_mu;
int g_cluster_fit[kMaxDevicesCached][4][9];  // max active clusters + 1 (0 = not yet queried)

}  // namespace

int sparse_cluster_size(int group, int units, int max_cluster)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesCached)
        return 1;
    const int gi = group == 1 ? 0 : group == 2 ? 1 : group == 4 ? 2 : 3;
    for (int C = 8; C >= 2; C >>= 1) {  // powers of two: each CTA owns 128 / C dims
        if (C > max_cluster)
            continue;
        int n;
        {
            std::lock_guard<std::mutex> lock(g_cluster_mu);
            n = g_cluster_fit[dev][gi][C] - 1;
        }
        if (n < 0) {
            n = max_active_clusters(group, C);
            std::lock_guard<std::mutex> lock(g_cluster_mu);
            g_cluster_fit[dev][gi][C] = n + 1;
        }
        if (n >= units)
            return C;
    }
    return 1;
}

size_t attention_smem_bytes() { return kSmemBytes; }

cudaError_t launch_attention(bool dense, int group, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                             const CUtensorMap &tm_q, const CUtensorMap &tm_kc,
                             const CUtensorMap &tm_vc, const AttnParams &p, int grid,
                             cudaStream_t stream)
{
#define SFI_ATTN_CASE(G)                                                                      \
    case G:                                                                                   \
        return dense ? launch_attn_t<G, true>(tm_k, tm_v, tm_q, tm_kc, tm_vc, p, grid, stream) \
                     : launch_attn_t<G, false>(tm_k, tm_v, tm_q, tm_kc, tm_vc, p, grid, stream);
    switch (group) {
        SFI_ATTN_CASE(1)
        SFI_ATTN_CASE(2)
        SFI_ATTN_CASE(4)
        SFI_ATTN_CASE(8)
    default:
        return cudaErrorInvalidValue;
    }
#undef SFI_ATTN_CASE
}

cudaError_t launch_evidence(const float *zbuf, const float2 *stats, float *f, const int32_t *seq_len,
                            const uint8_t *active, int n_layers, int batch, int n_kv_heads, int group,
                            int capacity, int max_len, cudaStream_t stream, int n_seq_active)
{
    const int units = n_layers * (n_seq_active > 0 ? n_seq_active : batch) * n_kv_heads;
    dim3 grid((max_len + 256 * kEvPer - 1) / (256 * kEvPer), units);
    if (grid.x == 0)
        grid.x = 1;
    switch (group) {
    case 1: return launch_pdl(evidence_kernel<1>, grid, dim3(256), 0, stream, zbuf, stats, f, seq_len, active, batch, n_kv_heads, capacity, n_seq_active);
    case 2: return launch_pdl(evidence_kernel<2>, grid, dim3(256), 0, stream, zbuf, stats, f, seq_len, active, batch, n_kv_heads, capacity, n_seq_active);
    case 4: return launch_pdl(evidence_kernel<4>, grid, dim3(256), 0, stream, zbuf, stats, f, seq_len, active, batch, n_kv_heads, capacity, n_seq_active);
    case 8: return launch_pdl(evidence_kernel<8>, grid, dim3(256), 0, stream, zbuf, stats, f, seq_len, active, batch, n_kv_heads, capacity, n_seq_active);
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------
// Fast step without a caller workspace.
//
// Some callers cannot allocate device memory at all -- for example a host framework that
// hands a plug-in only its input and output buffers, or a real-time decode loop that must
// never call cudaMalloc (it can synchronise the device). For them the fast step keeps its
// split-KV scratch (partials and tickets) in this file-scope array, which every GPU that
// loads the library holds until the process exits. In host code the array's name is only
// a host-side stand-in, so its device address is looked up once per device.

constexpr size_t kStaticPartialBytes =
    static_cast<size_t>(2) * kStaticMaxCtas * kPartialFloats(8) * sizeof(float);
constexpr size_t kStaticScratchBytes = kStaticPartialBytes + kStaticMaxUnits * sizeof(int);

static __device__ __align__(256) unsigned char g_sfi_static_scratch[kStaticScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void *g_static_addr[kMaxDevices] = {};

// Device address of g_sfi_static_scratch on the current device (set up on first use).
cudaError_t static_scratch(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (g_static_addr[dev] == nullptr) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_sfi_static_scratch);
        if (e != cudaSuccess)
            return e;
        g_static_addr[dev] = ptr;
    }
    *out = g_static_addr[dev];
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_sparse_static(int group, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                 const CUtensorMap &tm_q, const CUtensorMap &tm_kc,
                                 const CUtensorMap &tm_vc, AttnParams p, int units, int grid,
                                 cudaStream_t stream)
{
    if (units > kStaticMaxUnits || grid > kStaticMaxCtas || group > 8)
        return cudaErrorInvalidValue;
    void *base = nullptr;
    cudaError_t e = static_scratch(&base);
    if (e != cudaSuccess)
        return e;
    p.partials = static_cast<float *>(base);
    p.tickets = reinterpret_cast<int *>(static_cast<unsigned char *>(base) + kStaticPartialBytes);
    // The tickets must start at zero; the array keeps whatever the previous call left.
    e = cudaMemsetAsync(p.tickets, 0, static_cast<size_t>(units) * sizeof(int), stream);
    if (e != cudaSuccess)
        return e;
    return launch_attention(false, group, tm_k, tm_v, tm_q, tm_kc, tm_vc, p, grid, stream);
}

}  // namespace sfi
