// sfi_internal.h -- declarations shared by the library's host code and its kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sfi {

constexpr int kHeadDim = 128;           // elements per K/V/Q row (256 bytes of bf16)
constexpr int kTile = 128;              // KV rows per attention tile (UMMA M)
constexpr int kStages = 3;              // shared-memory ring depth of the attention kernels
constexpr int kMaxBatch = 256;
constexpr int kAttnThreads = 192;       // warp 0 TMA, warp 1 MMA, warps 2-5 softmax/epilogue
constexpr int kSelectThreads = 1024;
constexpr uint64_t kWaitTimeoutNs = 1000000000ull;  // bounded pipeline waits: 1 s
// split-KV partial: 128 x G unnormalised outputs (dim-major), then per head the running max
// and the weight sum (base-2 logits); 16-byte aligned for G >= 2 (the merge reads it in
// 16-byte pieces for G >= 4)
constexpr int kPartialFloats(int G) { return G * kHeadDim + 2 * G; }

// Everything the attention kernels read besides the tensor maps.
struct AttnParams {
    int n_layers, batch, n_kv_heads, group;
    int capacity, page_size, n_pages, max_pages;
    int max_len;
    const int32_t *page_table;
    const int32_t *seq_len;
    const uint8_t *active;
    uint32_t *err;
    // sparse step
    const int32_t *comp_rows;   // packed rows per unit
    const int32_t *sel_cnt;     // selected rows per unit
    int comp_cap;               // n_sink + n_select: packed-buffer rows per unit
    int n_window;
    int n_cbox;                 // 64-row boxes of the packed region per unit
    int n_wbox;                 // 16-row boxes of the window region per unit
    int tiles_per_unit;         // sparse: ceil((64 n_cbox + 16 n_wbox) / 128)
    int cluster;                // sparse: CTAs per unit in one thread-block cluster (1 = none)
    // sparse step with the append fused in (k_new != null): each active sequence's new K/V
    // rows are written at position seq_len[b] and attended, and the last CTA to have read
    // seq_len advances it.
    const void *k_new, *v_new;  // bf16 [units][128]
    void *k_cache, *v_cache;    // the cache the tensor maps view
    int *append_counter;        // CTAs that have read seq_len; zero between launches
    int test_stall;             // test hook: CTA 0 waits on a barrier that never completes
    // outputs and workspace
    void *out;
    int out_fp32;
    float *zbuf;                // dense: base-2 logits [units][capacity][G] (or null)
    float2 *stats;              // dense: (max, sum) of base-2 logits per (unit, head)
    float *partials;            // [2 * gridDim.x][kPartialFloats(G)]
    int *tickets;               // [units]
    float scale_log2;           // log2(e) / sqrt(128)
};

struct SelectParams {
    const float *f;             // [units][capacity]
    int capacity, batch, n_kv_heads;
    int n_units;                // units launched (all, or the active sequences' with n_seq_active)
    int max_len;                // bound of every seq_len entry (a longer one: SFI_DEVERR_LENGTH)
    const int32_t *seq_len;
    const uint8_t *active;
    int n_sink, n_window, n_select, prior_tau;
    double lambda;
    int32_t *sel_idx;           // [units][n_select]
    int32_t *sel_cnt;           // [units]
    int staged;                 // candidates' evidence copied to shared memory (see kStageCap)
    int cluster;                // > 1: CTAs per unit in one cluster (select_cluster_size)
    uint32_t *err;              // device error word
    // > 0: the grid covers only the units of the first n_seq_active sequences with active[b]
    // set, per layer in order (the caller knows how many are active); 0: every unit
    int n_seq_active;
    // clustered Selector, group of 4: with zbuf set the evidence of each candidate is computed
    // here from the dense step's base-2 logits and merged statistics (as the evidence pass
    // does) and written to f_out; f is then not read
    const float *zbuf;          // [units][capacity][4]
    const float2 *stats;        // [units][4]
    float *f_out;               // [units][capacity]
};
// The Selector stages a unit's evidence in shared memory when it has at most this many
// candidates (plus alignment slack); larger units stream it from global memory.
constexpr int kStageCap = 36864;

struct RefineParams {
    const float *f;             // evidence [units][capacity]
    const float *key_norms;     // [units][capacity] or null
    float *refined;             // [units][capacity]
    int capacity, batch, n_kv_heads;
    const int32_t *seq_len;
    const uint8_t *active;
    int n_sink, n_window, prior_tau;
    double lambda;
    int geometric;
    float norm_nu;
    int nms_radius;
    float nms_gamma;
    float nms_delta;
    float excl_mu;
};

// Launchers (return the cudaGetLastError() of the launch).
cudaError_t launch_refine(const RefineParams &p, int n_layer_seq, int max_cand,
                          cudaStream_t stream);
cudaError_t launch_key_norms(const void *k, float *norms, const int32_t *seq_len,
                             const uint8_t *active, int n_layers, int batch, int n_kv_heads,
                             int capacity, int page_size, int n_pages, int max_pages,
                             const int32_t *page_table, int max_len, uint32_t *err,
                             cudaStream_t stream);
cudaError_t launch_attention(bool dense, int group, const CUtensorMap &tm_k,
                             const CUtensorMap &tm_v, const CUtensorMap &tm_q,
                             const CUtensorMap &tm_kc, const CUtensorMap &tm_vc,
                             const AttnParams &p, int grid, cudaStream_t stream);
// Largest cluster size (8, 4 or 2, at most max_cluster) for which `units` clusters of the
// sparse kernel can be resident at once (1 when none fits).
int sparse_cluster_size(int group, int units, int max_cluster);
cudaError_t launch_evidence(const float *zbuf, const float2 *stats, float *f,
                            const int32_t *seq_len, const uint8_t *active, int n_layers,
                            int batch, int n_kv_heads, int group, int capacity, int max_len,
                            cudaStream_t stream, int n_seq_active = 0);
cudaError_t launch_select(const SelectParams &p, cudaStream_t stream);
// Clustered Selector: the largest cluster size (4 or 2, at most max_cluster) that can be
// launched on this device (1 when none can); and the most candidates one of its CTAs can
// stage.
int select_cluster_size(int max_cluster);
int select_cluster_key_cap();
cudaError_t launch_append(const void *k_new, const void *v_new, void *k, void *v,
                          int32_t *seq_len, const uint8_t *active, const int32_t *page_table,
                          int n_layers, int batch, int n_kv_heads, int capacity, int page_size,
                          int n_pages, int max_pages, uint32_t *err, cudaStream_t stream);
cudaError_t launch_compact(const void *k, const void *v, void *kc, void *vc,
                           const int32_t *sel_idx, const int32_t *sel_cnt, int32_t *rows,
                           const int32_t *seq_len, const uint8_t *active,
                           const int32_t *page_table, int n_layers, int batch, int n_kv_heads,
                           int capacity, int page_size, int n_pages, int max_pages, int n_sink,
                           int n_select, uint32_t *err, cudaStream_t stream,
                           int n_seq_active = 0);

size_t attention_smem_bytes();
// Fast-step attention with its split-KV scratch in a library-owned device array instead of
// a caller workspace (see sfi_sparse_decode_attn_static). p.partials and p.tickets are
// filled in here. Limits: at most kStaticMaxUnits units; the grid is capped at
// kStaticMaxCtas CTAs.
constexpr int kStaticMaxCtas = 256;
constexpr int kStaticMaxUnits = 16384;
cudaError_t launch_sparse_static(int group, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                 const CUtensorMap &tm_q, const CUtensorMap &tm_kc,
                                 const CUtensorMap &tm_vc, AttnParams p, int units, int grid,
                                 cudaStream_t stream);

}  // namespace sfi
