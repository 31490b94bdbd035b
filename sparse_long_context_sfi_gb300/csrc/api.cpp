// api.cpp -- the extern "C" entry points declared in include/sfi.h: argument checks,
// workspace layout, TMA tensor-map encoding and kernel launches. No allocation, no
// synchronisation (except sfi_read_error), no state beyond the resolved driver entry point.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "sfi.h"
#include "sfi_internal.h"

using namespace sfi;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D bf16 view [rows][128] with 256-byte rows; box = 64 columns x box_rows rows, 128-byte
// swizzle (the canonical K-major / MN-major operand layout of the UMMA descriptors).
bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint32_t box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn || rows == 0)
        return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), rows};
    const cuuint64_t strides[1] = {kHeadDim * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

sfi_status check_kv(const sfi_kv_cache *kv)
{
    if (!kv || !kv->k || !kv->v || !kv->seq_len || !kv->err)
        return SFI_ERR_INVALID_ARG;
    if (kv->n_layers < 1 || kv->batch < 1 || kv->n_kv_heads < 1 || kv->n_q_heads < 1)
        return SFI_ERR_INVALID_ARG;
    if (kv->head_dim != kHeadDim || kv->batch > kMaxBatch)
        return SFI_ERR_UNSUPPORTED;
    if (kv->n_q_heads % kv->n_kv_heads != 0)
        return SFI_ERR_INVALID_ARG;
    const int g = kv->n_q_heads / kv->n_kv_heads;
    if (g != 1 && g != 2 && g != 4 && g != 8)
        return SFI_ERR_UNSUPPORTED;
    if (!aligned16(kv->k) || !aligned16(kv->v))
        return SFI_ERR_INVALID_ARG;
    if (kv->max_len < 0 || kv->capacity < 1)
        return SFI_ERR_INVALID_ARG;
    if (kv->page_size != 0) {
        if (kv->page_size != 16)
            return SFI_ERR_UNSUPPORTED;
        if (!kv->page_table || kv->n_pages < 1 || kv->max_pages_per_seq < 1 ||
            kv->capacity != kv->max_pages_per_seq * kv->page_size)
            return SFI_ERR_INVALID_ARG;
    }
    if (kv->max_len > kv->capacity)
        return SFI_ERR_CAPACITY;
    const long long units = 1LL * kv->n_layers * kv->batch * kv->n_kv_heads;
    const long long rows = kv->page_size ? 1LL * kv->n_layers * kv->n_pages * kv->n_kv_heads * 16
                                         : units * kv->capacity;
    if (units > 65535 || rows >= (1LL << 31))
        return SFI_ERR_UNSUPPORTED;
    return SFI_OK;
}

sfi_status check_budget(const sfi_budget *bd)
{
    if (!bd || bd->n_sink < 0 || bd->n_window < 1 || bd->n_select < 0 || bd->prior_tau < 1)
        return SFI_ERR_INVALID_ARG;
    if ((bd->prior_tau & (bd->prior_tau - 1)) != 0 || !(bd->lambda >= 0.0 && bd->lambda <= 1.0))
        return SFI_ERR_INVALID_ARG;
    if (bd->n_sink + bd->n_select < 1)
        return SFI_ERR_INVALID_ARG;
    return SFI_OK;
}

int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
    size_t tickets_dense, tickets_sparse, append_ctr, append_ctr_dense, stats, part_dense,
        part_sparse, zbuf, total;
};

WsLayout ws_layout(const sfi_kv_cache *kv, int sms)
{
    const size_t units = static_cast<size_t>(kv->n_layers) * kv->batch * kv->n_kv_heads;
    const int g = kv->n_q_heads / kv->n_kv_heads;
    const size_t part = static_cast<size_t>(2) * sms * kPartialFloats(g) * sizeof(float);
    WsLayout w;
    size_t o = 0;
    w.tickets_dense = o;  o = align256(o + units * sizeof(int));
    w.tickets_sparse = o; o = align256(o + units * sizeof(int));
    w.append_ctr = o;     o = align256(o + sizeof(int));
    w.append_ctr_dense = o; o = align256(o + sizeof(int));
    w.stats = o;          o = align256(o + units * g * sizeof(float2));
    w.part_dense = o;     o = align256(o + part);
    w.part_sparse = o;    o = align256(o + part);
    w.zbuf = o;           o = align256(o + units * static_cast<size_t>(kv->capacity) * g * sizeof(float));
    w.total = o;
    return w;
}

cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

// Timing events: recorded as external event nodes while the stream is being captured
// (so graph replays time the kernel), as plain records otherwise.
cudaError_t record_event(cudaEvent_t e, cudaStream_t s)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t err = cudaStreamIsCapturing(s, &cs);
    if (err != cudaSuccess)
        return err;
    return cudaEventRecordWithFlags(e, s, cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal
                                                                              : cudaEventRecordDefault);
}

sfi_status launch_status(cudaError_t e) { return e == cudaSuccess ? SFI_OK : SFI_ERR_CUDA; }

// One-shot test hook of sfi_test_inject_stall: consumed by the next attention launch.
std::atomic<int> g_test_stall{0};

void fill_common(AttnParams &p, const sfi_kv_cache *kv, const uint8_t *active)
{
    std::memset(&p, 0, sizeof p);
    p.n_layers = kv->n_layers;
    p.batch = kv->batch;
    p.n_kv_heads = kv->n_kv_heads;
    p.group = kv->n_q_heads / kv->n_kv_heads;
    p.capacity = kv->capacity;
    p.page_size = kv->page_size;
    p.n_pages = kv->n_pages;
    p.max_pages = kv->max_pages_per_seq;
    p.max_len = kv->max_len;
    p.page_table = kv->page_table;
    p.seq_len = kv->seq_len;
    p.active = active;
    p.err = kv->err;
    p.scale_log2 = static_cast<float>(1.4426950408889634074 / std::sqrt(static_cast<double>(kHeadDim)));
}

uint64_t cache_rows(const sfi_kv_cache *kv)
{
    if (kv->page_size)
        return static_cast<uint64_t>(kv->n_layers) * kv->n_pages * kv->n_kv_heads * kv->page_size;
    return static_cast<uint64_t>(kv->n_layers) * kv->batch * kv->n_kv_heads * kv->capacity;
}

// ws_kv/unit0: the descriptor whose workspace layout `ws` follows and the first of its units
// that kv covers (a one-layer view of a larger cache keeps the per-unit regions of the whole
// cache, so the tickets and counters of every other launch stay where they are).
// n_seq_active > 0: exactly that many sequences have active[b] set (the evidence pass then
// launches only their units). k_new/v_new: the append of the active sequences' new rows is
// fused in, as in the fast step (kv->max_len then bounds the lengths before the append; whole
// caches only: the last CTA advances seq_len).
sfi_status dense_impl(const sfi_kv_cache *kv, const void *q, void *out, int32_t out_fp32,
                      float *scores_f, const uint8_t *active, void *ws, size_t ws_bytes,
                      void *stream, cudaEvent_t e0, cudaEvent_t e1,
                      const sfi_kv_cache *ws_kv = nullptr, long long unit0 = 0,
                      int n_seq_active = 0, const void *k_new = nullptr,
                      const void *v_new = nullptr, bool evidence = true)
{
    sfi_status st = check_kv(kv);
    if (st != SFI_OK)
        return st;
    if (!q || !out || !aligned16(q))
        return SFI_ERR_INVALID_ARG;
    const bool fused = k_new != nullptr || v_new != nullptr;
    if (fused) {
        if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new) || ws_kv)
            return SFI_ERR_INVALID_ARG;
        if (kv->max_len + 1 > kv->capacity)
            return SFI_ERR_CAPACITY;
    }
    const int len_bound = kv->max_len + (fused ? 1 : 0);  // lengths after the append
    const int sms = sm_count();
    if (sms <= 0)
        return SFI_ERR_CUDA;
    const WsLayout w = ws_layout(ws_kv ? ws_kv : kv, sms);
    if (!ws || ws_bytes < w.total || (reinterpret_cast<uintptr_t>(ws) & 255u))
        return SFI_ERR_WORKSPACE;
    if (len_bound == 0)
        return SFI_OK;
    char *base = static_cast<char *>(ws);
    AttnParams p;
    fill_common(p, kv, active);
    const int g = p.group;
    if (fused) {
        p.k_new = k_new;
        p.v_new = v_new;
        p.k_cache = kv->k;
        p.v_cache = kv->v;
        p.append_counter = reinterpret_cast<int *>(base + w.append_ctr_dense);
    }
    p.out = out;
    p.out_fp32 = out_fp32 ? 1 : 0;
    p.zbuf = scores_f ? reinterpret_cast<float *>(base + w.zbuf) +
                            unit0 * static_cast<long long>(kv->capacity) * g
                      : nullptr;
    p.test_stall = g_test_stall.exchange(0);
    p.stats = reinterpret_cast<float2 *>(base + w.stats) + unit0 * g;
    p.partials = reinterpret_cast<float *>(base + w.part_dense);
    p.tickets = reinterpret_cast<int *>(base + w.tickets_dense) + unit0;
    const long long units = 1LL * kv->n_layers * kv->batch * kv->n_kv_heads;
    CUtensorMap tk, tv, tq;
    const uint32_t box = kv->page_size ? 16u : static_cast<uint32_t>(kTile);
    if (!make_map(&tk, kv->k, cache_rows(kv), box) || !make_map(&tv, kv->v, cache_rows(kv), box) ||
        !make_map(&tq, q, static_cast<uint64_t>(units) * g, static_cast<uint32_t>(g)))
        return SFI_ERR_CUDA;
    const long long t_upper = units * ((len_bound + kTile - 1) / kTile);
    const int grid = static_cast<int>(t_upper < sms ? t_upper : sms);
    if (e0 && record_event(e0, as_stream(stream)) != cudaSuccess)
        return SFI_ERR_CUDA;
    cudaError_t e = launch_attention(true, g, tk, tv, tq, tk, tv, p, grid, as_stream(stream));
    if (e != cudaSuccess)
        return SFI_ERR_CUDA;
    if (e1 && record_event(e1, as_stream(stream)) != cudaSuccess)
        return SFI_ERR_CUDA;
    // (evidence false: the logits and statistics are left for the Selector, which computes
    // the evidence itself)
    if (scores_f && evidence) {
        e = launch_evidence(p.zbuf, p.stats, scores_f, kv->seq_len, active, kv->n_layers,
                            kv->batch, kv->n_kv_heads, g, kv->capacity, len_bound,
                            as_stream(stream),
                            (active && n_seq_active > 0 && n_seq_active < kv->batch) ? n_seq_active : 0);
        if (e != cudaSuccess)
            return SFI_ERR_CUDA;
    }
    return SFI_OK;
}

// The fast step; with k_new/v_new given, the append of the new rows is fused in (kv->max_len
// then bounds the lengths before the append).
sfi_status sparse_impl(const sfi_kv_cache *kv, const sfi_sparse_mem *mem,
                       const sfi_budget *budget, const void *q, void *out, int32_t out_fp32,
                       const uint8_t *active, void *ws, size_t ws_bytes, void *stream,
                       cudaEvent_t e0, cudaEvent_t e1, const void *k_new = nullptr,
                       const void *v_new = nullptr)
{
    sfi_status st = check_kv(kv);
    if (st != SFI_OK)
        return st;
    if ((st = check_budget(budget)) != SFI_OK)
        return st;
    if (!mem || !mem->kc || !mem->vc || !mem->sel_cnt || !mem->rows || !q || !out ||
        !aligned16(q) || !aligned16(mem->kc) || !aligned16(mem->vc))
        return SFI_ERR_INVALID_ARG;
    const bool fused = k_new != nullptr || v_new != nullptr;
    if (fused) {
        if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))
            return SFI_ERR_INVALID_ARG;
        if (kv->max_len + 1 > kv->capacity)
            return SFI_ERR_CAPACITY;
    }
    const int sms = sm_count();
    if (sms <= 0)
        return SFI_ERR_CUDA;
    const WsLayout w = ws_layout(kv, sms);
    if (!ws || ws_bytes < w.total || (reinterpret_cast<uintptr_t>(ws) & 255u))
        return SFI_ERR_WORKSPACE;
    char *base = static_cast<char *>(ws);
    AttnParams p;
    fill_common(p, kv, active);
    p.out = out;
    p.out_fp32 = out_fp32 ? 1 : 0;
    p.partials = reinterpret_cast<float *>(base + w.part_sparse);
    p.tickets = reinterpret_cast<int *>(base + w.tickets_sparse);
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_cache = kv->k;
    p.v_cache = kv->v;
    p.append_counter = reinterpret_cast<int *>(base + w.append_ctr);
    p.test_stall = g_test_stall.exchange(0);
    p.comp_rows = mem->rows;
    p.sel_cnt = mem->sel_cnt;
    p.comp_cap = budget->n_sink + budget->n_select;
    p.n_window = budget->n_window;
    p.n_cbox = (p.comp_cap + 63) / 64;
    p.n_wbox = (budget->n_window + 15) / 16 + (kv->page_size ? 1 : 0);
    p.tiles_per_unit = (64 * p.n_cbox + 16 * p.n_wbox + kTile - 1) / kTile;
    const int g = p.group;
    const long long units = 1LL * kv->n_layers * kv->batch * kv->n_kv_heads;
    CUtensorMap tk, tv, tq, tkc, tvc;
    if (!make_map(&tk, kv->k, cache_rows(kv), 16u) || !make_map(&tv, kv->v, cache_rows(kv), 16u) ||
        !make_map(&tq, q, static_cast<uint64_t>(units) * g, static_cast<uint32_t>(g)) ||
        !make_map(&tkc, mem->kc, static_cast<uint64_t>(units) * p.comp_cap, 64u) ||
        !make_map(&tvc, mem->vc, static_cast<uint64_t>(units) * p.comp_cap, 64u))
        return SFI_ERR_CUDA;
    // Few units: a cluster of up to 8 CTAs per unit (one unit per cluster, partials merged
    // in distributed shared memory). Otherwise one CTA per SM over contiguous tile ranges.
    int cluster = 1;
    if (units * 2 <= sms && g <= 4) {
        long long cmax = sms / units;
        cmax = cmax < 8 ? cmax : 8;
        cmax = cmax < p.tiles_per_unit ? cmax : p.tiles_per_unit;
        if (cmax >= 2)
            cluster = sparse_cluster_size(g, static_cast<int>(units), static_cast<int>(cmax));
    }
    p.cluster = cluster;
    const long long t_upper = units * p.tiles_per_unit;
    const int grid = cluster > 1 ? static_cast<int>(units) * cluster
                                 : static_cast<int>(t_upper < sms ? t_upper : sms);
    if (e0 && record_event(e0, as_stream(stream)) != cudaSuccess)
        return SFI_ERR_CUDA;
    if (launch_attention(false, g, tk, tv, tq, tkc, tvc, p, grid, as_stream(stream)) != cudaSuccess)
        return SFI_ERR_CUDA;
    if (e1 && record_event(e1, as_stream(stream)) != cudaSuccess)
        return SFI_ERR_CUDA;
    return SFI_OK;
}

// A cache descriptor and packed memory restricted to layers [l, l + nl) (base pointers
// offset by whole layers; every per-unit array is laid out layer-major).
void layer_views(const sfi_kv_cache *kv, const sfi_budget *budget, const sfi_sparse_mem *mem,
                 int l, int nl, sfi_kv_cache *kl, sfi_sparse_mem *ml)
{
    const size_t units = static_cast<size_t>(kv->batch) * kv->n_kv_heads;
    const size_t rows = kv->page_size ? static_cast<size_t>(kv->n_pages) * kv->n_kv_heads * 16
                                      : units * kv->capacity;
    const size_t comp = static_cast<size_t>(budget->n_sink + budget->n_select);
    *kl = *kv;
    kl->n_layers = nl;
    kl->k = static_cast<char *>(kv->k) + l * rows * kHeadDim * 2;
    kl->v = static_cast<char *>(kv->v) + l * rows * kHeadDim * 2;
    *ml = *mem;
    ml->kc = static_cast<char *>(mem->kc) + l * units * comp * kHeadDim * 2;
    ml->vc = static_cast<char *>(mem->vc) + l * units * comp * kHeadDim * 2;
    ml->sel_idx = mem->sel_idx + l * units * budget->n_select;
    ml->sel_cnt = mem->sel_cnt + l * units;
    ml->rows = mem->rows + l * units;
}

}  // namespace

extern "C" {

const char *sfi_status_string(sfi_status s)
{
    switch (s) {
    case SFI_OK: return "ok";
    case SFI_ERR_INVALID_ARG: return "invalid argument";
    case SFI_ERR_UNSUPPORTED: return "unsupported shape";
    case SFI_ERR_CAPACITY: return "length bound exceeds capacity";
    case SFI_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case SFI_ERR_CUDA: return "CUDA error";
    case SFI_ERR_DEVICE: return "device error word set";
    }
    return "unknown status";
}

const char *sfi_version(void) { return "sfi-gb300 0.1 (sm_103a, tcgen05/TMA)"; }

size_t sfi_workspace_bytes(const sfi_kv_cache *kv, const sfi_budget *budget)
{
    (void)budget;
    if (check_kv(kv) != SFI_OK)
        return 0;
    const int sms = sm_count();
    if (sms <= 0)
        return 0;
    return ws_layout(kv, sms).total;
}

sfi_status sfi_workspace_init(void *ws, size_t ws_bytes, void *stream)
{
    if (!ws || ws_bytes == 0)
        return SFI_ERR_WORKSPACE;
    return launch_status(cudaMemsetAsync(ws, 0, ws_bytes, as_stream(stream)));
}

sfi_status sfi_append_kv(const sfi_kv_cache *kv, const void *k_new, const void *v_new,
                         const uint8_t *active, void *stream)
{
    sfi_status st = check_kv(kv);
    if (st != SFI_OK)
        return st;
    if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))
        return SFI_ERR_INVALID_ARG;
    if (kv->max_len + 1 > kv->capacity)
        return SFI_ERR_CAPACITY;
    return launch_status(launch_append(k_new, v_new, kv->k, kv->v, kv->seq_len, active,
                                       kv->page_table, kv->n_layers, kv->batch, kv->n_kv_heads,
                                       kv->capacity, kv->page_size, kv->n_pages,
                                       kv->max_pages_per_seq, kv->err, as_stream(stream)));
}

sfi_status sfi_dense_decode_attn(const sfi_kv_cache *kv, const void *q, void *out,
                                 int32_t out_fp32, float *scores_f, const uint8_t *active,
                                 void *ws, size_t ws_bytes, void *stream)
{
    return dense_impl(kv, q, out, out_fp32, scores_f, active, ws, ws_bytes, stream, nullptr,
                      nullptr);
}

// How sfi_select runs for these arguments: the units it launches, whether the evidence is
// staged in shared memory, and the CTAs per unit (1: one CTA per unit; > 1: clustered).
struct SelectShape {
    int n_seq_active, n_units, staged, cluster;
};

static SelectShape select_shape(const sfi_kv_cache *kv, const float *scores_f,
                                const sfi_budget *budget, const uint8_t *active, int n_seq_active)
{
    SelectShape sh;
    sh.n_seq_active = (active && n_seq_active > 0 && n_seq_active < kv->batch) ? n_seq_active : 0;
    sh.n_units = kv->n_layers * (sh.n_seq_active > 0 ? sh.n_seq_active : kv->batch) * kv->n_kv_heads;
    // Stage in shared memory when every unit's candidates (with up to 3 values of alignment
    // slack on either side) fit, and the copy's tail stays inside the unit's row.
    const long long bound = static_cast<long long>(kv->max_len) - budget->n_window - budget->n_sink;
    const bool stageable = aligned16(scores_f) &&
                           static_cast<long long>(kv->max_len) - budget->n_window + 3 <= kv->capacity;
    sh.staged = (stageable && bound + 3 <= kStageCap) ? 1 : 0;
    // A unit's candidates split over a cluster of CTAs (each stages its share) when they fit.
    sh.cluster = 1;
    if (stageable) {
        const int C = select_cluster_size(4);
        const long long ctas = static_cast<long long>(sh.n_units) * C;
        if (C > 1 && (bound + C - 1) / C <= select_cluster_key_cap() && ctas <= 2LL * sm_count())
            sh.cluster = C;  // at most about two waves of CTAs
    }
    return sh;
}

// Whether sfi_decode_run's slow step leaves the evidence to the Selector (clustered, group of
// 4): one launch fewer, the evidence computed as the Selector stages its candidates.
static bool select_fuses_evidence(const sfi_kv_cache *kv, const float *scores_f,
                                  const sfi_budget *budget, const uint8_t *active, int n_seq_active)
{
    return kv->n_q_heads == 4 * kv->n_kv_heads &&
           select_shape(kv, scores_f, budget, active, n_seq_active).cluster > 1;
}

// sfi_select, with n_seq_active > 0 when the caller knows that exactly that many sequences
// have active[b] set (sfi_decode_run's slow subsets): the launch then covers only their units,
// which lets a small subset take the clustered Selector. ev_ws: the workspace whose logits
// and statistics the preceding dense launch (run without its evidence pass, whole-cache view)
// left: the clustered Selector then computes the evidence itself and writes it to scores_f
// (group of 4; the caller checked the shape with select_shape).
static sfi_status select_impl(const sfi_kv_cache *kv, const float *scores_f,
                              const sfi_budget *budget, const sfi_sparse_mem *mem,
                              const uint8_t *active, int n_seq_active, void *stream,
                              void *ev_ws = nullptr)
{
    sfi_status st = check_kv(kv);
    if (st != SFI_OK)
        return st;
    if ((st = check_budget(budget)) != SFI_OK)
        return st;
    if (!scores_f || !mem || !mem->sel_idx || !mem->sel_cnt)
        return SFI_ERR_INVALID_ARG;
    const SelectShape sh = select_shape(kv, scores_f, budget, active, n_seq_active);
    SelectParams p;
    std::memset(&p, 0, sizeof p);
    p.f = scores_f;
    p.capacity = kv->capacity;
    p.batch = kv->batch;
    p.n_kv_heads = kv->n_kv_heads;
    p.n_seq_active = sh.n_seq_active;
    p.n_units = sh.n_units;
    p.seq_len = kv->seq_len;
    p.max_len = kv->max_len;
    p.active = active;
    p.n_sink = budget->n_sink;
    p.n_window = budget->n_window;
    p.n_select = budget->n_select;
    p.prior_tau = budget->prior_tau;
    p.lambda = budget->lambda;
    p.sel_idx = mem->sel_idx;
    p.sel_cnt = mem->sel_cnt;
    p.err = kv->err;
    p.staged = sh.staged;
    p.cluster = sh.cluster;
    if (ev_ws) {
        if (sh.cluster <= 1 || kv->n_q_heads != 4 * kv->n_kv_heads)
            return SFI_ERR_INVALID_ARG;
        const WsLayout w = ws_layout(kv, sm_count());
        char *base = static_cast<char *>(ev_ws);
        p.zbuf = reinterpret_cast<const float *>(base + w.zbuf);
        p.stats = reinterpret_cast<const float2 *>(base + w.stats);
        p.f_out = const_cast<float *>(scores_f);
    }
    return launch_status(launch_select(p, as_stream(stream)));
}

sfi_status sfi_select(const sfi_kv_cache *kv, const float *scores_f, const sfi_budget *budget,
                      const sfi_sparse_mem *mem, const uint8_t *active, void *stream)
{
    return select_impl(kv, scores_f, budget, mem, active, 0, stream);
}

sfi_status sfi_key_norms(const sfi_kv_cache *kv, float *norms, const uint8_t *active,
                         void *stream)
{
    sfi_status st = check_kv(kv);
    if (st != SFI_OK)
        return st;
    if (!norms)
        return SFI_ERR_INVALID_ARG;
    return launch_status(launch_key_norms(kv->k, norms, kv->seq_len, active, kv->n_layers,
                                          kv->batch, kv->n_kv_heads, kv->capacity, kv->page_size,
                                          kv->n_pages, kv->max_pages_per_seq, kv->page_table,
                                          kv->max_len, kv->err, as_stream(stream)));
}

sfi_status sfi_refine_scores(const sfi_kv_cache *kv, const float *scores_f,
                             const float *key_norms, const sfi_budget *budget, float *refined,
                             const uint8_t *active, void *stream)
{
    sfi_status st = check_kv(kv);
    if (st != SFI_OK)
        return st;
    if ((st = check_budget(budget)) != SFI_OK)
        return st;
    if (!scores_f || !refined || budget->nms_radius < 0 ||
        !(budget->nms_gamma >= 0.f && budget->nms_gamma <= 1.f) || !(budget->nms_delta >= 0.f) ||
        !(budget->excl_mu >= 0.f && budget->excl_mu <= 1.f) || !(budget->norm_nu >= 0.f) ||
        (budget->norm_nu > 0.f && !key_norms))
        return SFI_ERR_INVALID_ARG;
    if (kv->n_kv_heads > 16)
        return SFI_ERR_UNSUPPORTED;
    RefineParams p;
    std::memset(&p, 0, sizeof p);
    p.f = scores_f;
    p.key_norms = key_norms;
    p.refined = refined;
    p.capacity = kv->capacity;
    p.batch = kv->batch;
    p.n_kv_heads = kv->n_kv_heads;
    p.seq_len = kv->seq_len;
    p.active = active;
    p.n_sink = budget->n_sink;
    p.n_window = budget->n_window;
    p.prior_tau = budget->prior_tau;
    p.lambda = budget->lambda;
    p.geometric = budget->geometric ? 1 : 0;
    p.norm_nu = budget->norm_nu;
    p.nms_radius = budget->nms_radius;
    p.nms_gamma = budget->nms_gamma;
    p.nms_delta = budget->nms_delta;
    p.excl_mu = budget->excl_mu;
    const int max_cand = kv->max_len - budget->n_window - budget->n_sink;
    return launch_status(
        launch_refine(p, kv->n_layers * kv->batch, max_cand > 0 ? max_cand : 1, as_stream(stream)));
}

// sfi_compact, with n_seq_active > 0 when exactly that many sequences have active[b] set (as
// for select_impl).
static sfi_status compact_impl(const sfi_kv_cache *kv, const sfi_budget *budget,
                               const sfi_sparse_mem *mem, const uint8_t *active,
                               int n_seq_active, void *stream)
{
    sfi_status st = check_kv(kv);
    if (st != SFI_OK)
        return st;
    if ((st = check_budget(budget)) != SFI_OK)
        return st;
    if (!mem || !mem->kc || !mem->vc || !mem->sel_idx || !mem->sel_cnt || !mem->rows ||
        !aligned16(mem->kc) || !aligned16(mem->vc))
        return SFI_ERR_INVALID_ARG;
    return launch_status(launch_compact(
        kv->k, kv->v, mem->kc, mem->vc, mem->sel_idx, mem->sel_cnt, mem->rows, kv->seq_len, active,
        kv->page_table, kv->n_layers, kv->batch, kv->n_kv_heads, kv->capacity, kv->page_size,
        kv->n_pages, kv->max_pages_per_seq, budget->n_sink, budget->n_select, kv->err,
        as_stream(stream),
        (active && n_seq_active > 0 && n_seq_active < kv->batch) ? n_seq_active : 0));
}

sfi_status sfi_compact(const sfi_kv_cache *kv, const sfi_budget *budget,
                       const sfi_sparse_mem *mem, const uint8_t *active, void *stream)
{
    return compact_impl(kv, budget, mem, active, 0, stream);
}

sfi_status sfi_sparse_decode_attn(const sfi_kv_cache *kv, const sfi_sparse_mem *mem,
                                  const sfi_budget *budget, const void *q, void *out,
                                  int32_t out_fp32, const uint8_t *active, void *ws,
                                  size_t ws_bytes, void *stream)
{
    return sparse_impl(kv, mem, budget, q, out, out_fp32, active, ws, ws_bytes, stream, nullptr,
                       nullptr);
}

sfi_status sfi_fast_decode_step(const sfi_kv_cache *kv, const sfi_sparse_mem *mem,
                                const sfi_budget *budget, const void *k_new, const void *v_new,
                                const void *q, void *out, int32_t out_fp32, const uint8_t *active,
                                void *ws, size_t ws_bytes, void *stream)
{
    if (!k_new || !v_new)
        return SFI_ERR_INVALID_ARG;
    return sparse_impl(kv, mem, budget, q, out, out_fp32, active, ws, ws_bytes, stream, nullptr,
                       nullptr, k_new, v_new);
}

sfi_status sfi_sparse_decode_attn_static(const sfi_kv_cache *kv, const sfi_sparse_mem *mem,
                                         const sfi_budget *budget, const void *q, void *out,
                                         int32_t out_fp32, const uint8_t *active, void *stream)
{
    sfi_status st = check_kv(kv);
    if (st != SFI_OK)
        return st;
    if ((st = check_budget(budget)) != SFI_OK)
        return st;
    if (!mem || !mem->kc || !mem->vc || !mem->sel_cnt || !mem->rows || !q || !out ||
        !aligned16(q) || !aligned16(mem->kc) || !aligned16(mem->vc))
        return SFI_ERR_INVALID_ARG;
    const long long units = 1LL * kv->n_layers * kv->batch * kv->n_kv_heads;
    if (units > kStaticMaxUnits)
        return SFI_ERR_CAPACITY;  // beyond the static scratch: use sfi_sparse_decode_attn
    const int sms = sm_count();
    if (sms <= 0)
        return SFI_ERR_CUDA;
    AttnParams p;
    fill_common(p, kv, active);
    p.out = out;
    p.out_fp32 = out_fp32 ? 1 : 0;
    p.comp_rows = mem->rows;
    p.sel_cnt = mem->sel_cnt;
    p.comp_cap = budget->n_sink + budget->n_select;
    p.n_window = budget->n_window;
    p.n_cbox = (p.comp_cap + 63) / 64;
    p.n_wbox = (budget->n_window + 15) / 16 + (kv->page_size ? 1 : 0);
    p.tiles_per_unit = (64 * p.n_cbox + 16 * p.n_wbox + kTile - 1) / kTile;
    const int g = p.group;
    CUtensorMap tk, tv, tq, tkc, tvc;
    if (!make_map(&tk, kv->k, cache_rows(kv), 16u) || !make_map(&tv, kv->v, cache_rows(kv), 16u) ||
        !make_map(&tq, q, static_cast<uint64_t>(units) * g, static_cast<uint32_t>(g)) ||
        !make_map(&tkc, mem->kc, static_cast<uint64_t>(units) * p.comp_cap, 64u) ||
        !make_map(&tvc, mem->vc, static_cast<uint64_t>(units) * p.comp_cap, 64u))
        return SFI_ERR_CUDA;
    long long grid = units * p.tiles_per_unit;
    if (grid > sms)
        grid = sms;
    if (grid > kStaticMaxCtas)
        grid = kStaticMaxCtas;
    return launch_status(launch_sparse_static(g, tk, tv, tq, tkc, tvc, p, static_cast<int>(units),
                                              static_cast<int>(grid), as_stream(stream)));
}

sfi_status sfi_schedule(int32_t steps, const uint8_t *mask, int32_t t_max, uint8_t *slow)
{
    if (steps < 0 || (steps > 0 && (!mask || !slow)))
        return SFI_ERR_INVALID_ARG;
    int32_t last = 0;
    for (int32_t t = 0; t < steps; ++t) {
        const bool s = t == 0 || mask[t - 1] != 0 || (t_max > 0 && t - last >= t_max);
        slow[t] = s ? 1 : 0;
        if (s)
            last = t;
    }
    return SFI_OK;
}

// One slow step with the layer-wise asynchronous pipeline (technical summary section 3,
// layer-wise overlap): attention and evidence of a group of layers on the main stream, then
// the Selector and compaction of that group on the side stream, forked after the group's
// evidence so that they run beside the attention of the next group; joined back at the end
// of the step. Groups of several layers keep each dense launch long enough to fill the GPU.
static sfi_status slow_step_layers(const sfi_kv_cache *k, const sfi_budget *budget,
                                   const sfi_sparse_mem *mem, const sfi_decode_plan *plan,
                                   const void *q, void *out, const uint8_t *m_slow, int n_slow_seq, void *ws,
                                   size_t ws_bytes, void *stream, cudaEvent_t e0, cudaEvent_t e1)
{
    cudaStream_t main_s = as_stream(stream), side = as_stream(plan->side_stream);
    cudaEvent_t fork = static_cast<cudaEvent_t>(plan->fork_event);
    cudaEvent_t join = static_cast<cudaEvent_t>(plan->join_event);
    const size_t units = static_cast<size_t>(k->batch) * k->n_kv_heads;
    const size_t q_layer = static_cast<size_t>(k->batch) * k->n_q_heads * kHeadDim;
    // layers per group: the plan's, or about a quarter of the layers
    int group = plan->pipeline_group > 0 ? plan->pipeline_group : (k->n_layers + 3) / 4;
    group = group < 1 ? 1 : (group > k->n_layers ? k->n_layers : group);
    if (e0 && record_event(e0, main_s) != cudaSuccess)
        return SFI_ERR_CUDA;
    sfi_status st = SFI_OK;
    bool forked = false;
    for (int l = 0; l < k->n_layers && st == SFI_OK; l += group) {
        const int nl = l + group <= k->n_layers ? group : k->n_layers - l;
        sfi_kv_cache kl;
        sfi_sparse_mem ml;
        layer_views(k, budget, mem, l, nl, &kl, &ml);
        const void *ql = static_cast<const char *>(q) + l * q_layer * 2;
        void *ol = static_cast<char *>(out) + l * q_layer * (plan->out_fp32 ? 4 : 2);
        float *fl = plan->scores_f + l * units * k->capacity;
        st = dense_impl(&kl, ql, ol, plan->out_fp32, fl, m_slow, ws, ws_bytes, stream, nullptr,
                        nullptr, k, static_cast<long long>(l) * units, n_slow_seq);
        if (st != SFI_OK)
            break;
        if (cudaEventRecord(fork, main_s) != cudaSuccess ||
            cudaStreamWaitEvent(side, fork, 0) != cudaSuccess) {
            st = SFI_ERR_CUDA;
            break;
        }
        forked = true;
        if ((st = select_impl(&kl, fl, budget, &ml, m_slow, n_slow_seq, plan->side_stream)) == SFI_OK)
            st = compact_impl(&kl, budget, &ml, m_slow, n_slow_seq, plan->side_stream);
    }
    // joined on every path once forked, so a stream capture around the call stays joinable
    if (forked && (cudaEventRecord(join, side) != cudaSuccess ||
                   cudaStreamWaitEvent(main_s, join, 0) != cudaSuccess) && st == SFI_OK)
        st = SFI_ERR_CUDA;
    if (st == SFI_OK && e1 && record_event(e1, main_s) != cudaSuccess)
        st = SFI_ERR_CUDA;
    return st;
}

sfi_status sfi_decode_run(const sfi_kv_cache *kv, const sfi_budget *budget,
                          const sfi_sparse_mem *mem, const sfi_decode_plan *plan, void *ws,
                          size_t ws_bytes, void *stream)
{
    sfi_status st = check_kv(kv);
    if (st != SFI_OK)
        return st;
    if ((st = check_budget(budget)) != SFI_OK)
        return st;
    if (!plan || !mem || plan->n_steps < 0 || !plan->slow || !plan->q || !plan->k_new ||
        !plan->v_new || !plan->out || !plan->scores_f || plan->len_start < 0)
        return SFI_ERR_INVALID_ARG;
    if (plan->len_start + plan->n_steps > kv->capacity)
        return SFI_ERR_CAPACITY;
    const bool conc_req = plan->concurrent_fast != 0 && !plan->dense_only;
    const bool pipe = plan->side_stream != nullptr && !plan->dense_only && !conc_req;
    if ((pipe || conc_req) && (!plan->side_stream || !plan->fork_event || !plan->join_event))
        return SFI_ERR_INVALID_ARG;
    const int B = kv->batch, g = kv->n_q_heads / kv->n_kv_heads;
    const size_t q_step = static_cast<size_t>(kv->n_layers) * B * kv->n_q_heads * kHeadDim;
    const size_t kv_step = static_cast<size_t>(kv->n_layers) * B * kv->n_kv_heads * kHeadDim;
    const size_t o_step = plan->out_per_step ? q_step * (plan->out_fp32 ? 4 : 2) : 0;
    (void)g;
    sfi_kv_cache k = *kv;
    for (int32_t t = 0; t < plan->n_steps; ++t) {
        const uint8_t *row = plan->slow + static_cast<size_t>(t) * B;
        int n_slow = 0;
        for (int b = 0; b < B; ++b)
            n_slow += row[b] ? 1 : 0;
        const bool mixed = n_slow != 0 && n_slow != B;
        if (mixed && !plan->masks && !plan->dense_only)
            return SFI_ERR_INVALID_ARG;
        const uint8_t *m_slow = mixed ? plan->masks + static_cast<size_t>(t) * 2 * B : nullptr;
        const uint8_t *m_fast = mixed ? m_slow + B : nullptr;
        const void *k_new = static_cast<const char *>(plan->k_new) + t * kv_step * 2;
        const void *v_new = static_cast<const char *>(plan->v_new) + t * kv_step * 2;
        // The new rows are appended inside the step's attention kernel: the fast sequences'
        // by the fast step, the slow sequences' by the dense step (kd: the dense launch's
        // cache view, whose max_len then bounds the lengths before the append). Only the
        // layer-wise pipeline's per-group dense launches append the slow sequences' rows
        // first.
        sfi_kv_cache kd = k;
        kd.max_len = plan->len_start + t;
        const bool sep_append = n_slow > 0 && pipe;
        if (sep_append) {
            st = sfi_append_kv(&kd, k_new, v_new, m_slow, stream);
            if (st != SFI_OK)
                return st;
            kd.max_len = plan->len_start + t + 1;
        }
        const void *kd_new = sep_append ? nullptr : k_new;
        const void *vd_new = sep_append ? nullptr : v_new;
        k.max_len = plan->len_start + t + 1;
        const void *q = static_cast<const char *>(plan->q) + t * q_step * 2;
        void *out = static_cast<char *>(plan->out) + t * o_step;
        cudaEvent_t e0 = plan->events ? static_cast<cudaEvent_t>(plan->events[2 * t]) : nullptr;
        cudaEvent_t e1 = plan->events ? static_cast<cudaEvent_t>(plan->events[2 * t + 1]) : nullptr;
        if (plan->dense_only) {
            if ((st = dense_impl(&kd, q, out, plan->out_fp32, nullptr, nullptr, ws, ws_bytes, stream,
                                 e0, e1, nullptr, 0, 0, kd_new, vd_new)) != SFI_OK)
                return st;
            continue;
        }
        if (mixed && conc_req) {
            // The slow subset's chain and the other sequences' fused fast step touch disjoint
            // sequences, cache rows, packed memory and workspace regions: the fast step runs
            // on the side stream beside the chain's Selector and packing, forked after the
            // chain's dense launch (and its evidence pass, when the Selector does not compute
            // the evidence itself). Both attention kernels take one CTA per SM and would
            // mostly queue behind each other; the Selector and packing leave the GPU largely
            // idle (forking before the dense launch, or splitting the SMs between the two by
            // bytes, was measured slower).
            cudaStream_t ms = as_stream(stream), ss = as_stream(plan->side_stream);
            cudaEvent_t fork = static_cast<cudaEvent_t>(plan->fork_event);
            cudaEvent_t join = static_cast<cudaEvent_t>(plan->join_event);
            const bool fev = select_fuses_evidence(&k, plan->scores_f, budget, m_slow, n_slow);
            if ((st = dense_impl(&kd, q, out, plan->out_fp32, plan->scores_f, m_slow, ws, ws_bytes,
                                 stream, e0, e1, nullptr, 0, n_slow, kd_new, vd_new, !fev)) != SFI_OK)
                return st;
            if (cudaEventRecord(fork, ms) != cudaSuccess || cudaStreamWaitEvent(ss, fork, 0) != cudaSuccess)
                return SFI_ERR_CUDA;
            sfi_kv_cache kf = k;
            kf.max_len = plan->len_start + t;  // the fused append's bound before appending
            st = sparse_impl(&kf, mem, budget, q, out, plan->out_fp32, m_fast, ws, ws_bytes,
                             plan->side_stream, nullptr, nullptr, k_new, v_new);
            // joined on every path once forked, so a stream capture around the call stays joinable
            if (cudaEventRecord(join, ss) != cudaSuccess && st == SFI_OK)
                st = SFI_ERR_CUDA;
            if (st == SFI_OK)
                st = select_impl(&k, plan->scores_f, budget, mem, m_slow, n_slow, stream,
                                 fev ? ws : nullptr);
            if (st == SFI_OK)
                st = compact_impl(&k, budget, mem, m_slow, n_slow, stream);
            if (cudaStreamWaitEvent(ms, join, 0) != cudaSuccess && st == SFI_OK)
                st = SFI_ERR_CUDA;
            if (st != SFI_OK)
                return st;
            continue;
        }
        if (n_slow > 0 && pipe) {
            if ((st = slow_step_layers(&k, budget, mem, plan, q, out, m_slow, mixed ? n_slow : 0, ws, ws_bytes,
                                       stream, e0, e1)) != SFI_OK)
                return st;
        } else if (n_slow > 0) {
            const int nsa = mixed ? n_slow : 0;
            const bool fev = select_fuses_evidence(&k, plan->scores_f, budget, m_slow, nsa);
            if ((st = dense_impl(&kd, q, out, plan->out_fp32, plan->scores_f, m_slow, ws, ws_bytes,
                                 stream, e0, e1, nullptr, 0, nsa, kd_new, vd_new, !fev)) != SFI_OK ||
                (st = select_impl(&k, plan->scores_f, budget, mem, m_slow, nsa, stream,
                                  fev ? ws : nullptr)) != SFI_OK ||
                (st = compact_impl(&k, budget, mem, m_slow, mixed ? n_slow : 0, stream)) != SFI_OK)
                return st;
        }
        if (n_slow < B) {
            k.max_len = plan->len_start + t;  // the fused append's bound before appending
            if ((st = sparse_impl(&k, mem, budget, q, out, plan->out_fp32, m_fast, ws, ws_bytes,
                                  stream, n_slow > 0 ? nullptr : e0, n_slow > 0 ? nullptr : e1,
                                  k_new, v_new)) != SFI_OK)
                return st;
        }
    }
    return SFI_OK;
}

sfi_status sfi_schedule_tokens(int32_t steps, const int32_t *tokens, const int32_t *trigger_ids,
                               int32_t n_trigger, int32_t t_max, uint8_t *slow)
{
    if (steps < 0 || n_trigger < 0 || (steps > 0 && (!tokens || !slow)) ||
        (n_trigger > 0 && !trigger_ids))
        return SFI_ERR_INVALID_ARG;
    int32_t last = 0;
    for (int32_t t = 0; t < steps; ++t) {
        bool trig = false;
        for (int32_t i = 0; t > 0 && i < n_trigger && !trig; ++i)
            trig = tokens[t - 1] == trigger_ids[i];
        const bool s = t == 0 || trig || (t_max > 0 && t - last >= t_max);
        slow[t] = s ? 1 : 0;
        if (s)
            last = t;
    }
    return SFI_OK;
}

sfi_status sfi_test_inject_stall(int32_t on)
{
    g_test_stall.store(on ? 1 : 0);
    return SFI_OK;
}

sfi_status sfi_read_error(const sfi_kv_cache *kv, uint32_t *bits, void *stream)
{
    if (!kv || !kv->err || !bits)
        return SFI_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    if (cudaMemcpyAsync(bits, kv->err, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return SFI_ERR_CUDA;
    return *bits ? SFI_ERR_DEVICE : SFI_OK;
}

sfi_status sfi_clear_error(const sfi_kv_cache *kv, void *stream)
{
    if (!kv || !kv->err)
        return SFI_ERR_INVALID_ARG;
    return launch_status(cudaMemsetAsync(kv->err, 0, sizeof(uint32_t), as_stream(stream)));
}

}  // extern "C"
