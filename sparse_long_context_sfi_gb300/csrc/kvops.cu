// kvops.cu -- KV-cache row movement for the SFI decode loop.
//   append:  every decode step writes the new token's K/V row at seq_len[b] (section 1 of
//            the gist.science technical summary: each step extends the history).
//   compact: after a slow step, packs the sink rows and the selected rows of each unit into
//            one contiguous buffer (section 3 of that summary, "Memory-Coalesced Sparse
//            Kernel"), so the fast step streams them sequentially.
// Both move 256-byte rows as 16 x 16-byte vectors per half-warp (coalesced 128-bit
// accesses); paged sources go through the page table with a range check.
#include "sfi_device.cuh"

namespace sfi {
namespace {

__global__ void __launch_bounds__(256) append_kernel(
    const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new, uint4 *__restrict__ k,
    uint4 *__restrict__ v, int32_t *__restrict__ seq_len, const uint8_t *__restrict__ active,
    const int32_t *__restrict__ page_table, int n_layers, int batch, int n_kv_heads, int capacity,
    int page_size, int n_pages, int max_pages, uint32_t *err)
{
    __shared__ int sh_ok, sh_pos, sh_page;
    const int b = blockIdx.x, tid = threadIdx.x;
    pdl_trigger();
    pdl_wait();
    if (active && !active[b])
        return;
    if (tid == 0) {
        const int pos = seq_len[b];
        int ok = pos >= 0 && pos < capacity;
        int page = 0;
        if (!ok)
            raise_error(err, 0x2u);  // SFI_DEVERR_CAPACITY
        if (ok && page_size > 0) {
            page = page_table[b * max_pages + pos / page_size];
            if (page < 0 || page >= n_pages) {
                raise_error(err, 0x1u);  // SFI_DEVERR_PAGE_RANGE
                ok = 0;
            }
        }
        sh_ok = ok;
        sh_pos = pos;
        sh_page = page;
    }
    __syncthreads();
    if (!sh_ok)
        return;
    const int pos = sh_pos, page = sh_page;
    const int rows = n_layers * n_kv_heads;
    const int per_tensor = rows * 16;
    for (int idx = tid; idx < 2 * per_tensor; idx += blockDim.x) {
        const int which = idx / per_tensor;
        const int rem = idx - which * per_tensor;
        const int rr = rem >> 4, ch = rem & 15;
        const int layer = rr / n_kv_heads, kvh = rr - layer * n_kv_heads;
        const size_t src = (static_cast<size_t>(layer * batch + b) * n_kv_heads + kvh) * 16 + ch;
        size_t dst_row;
        if (page_size == 0)
            dst_row = (static_cast<size_t>(layer * batch + b) * n_kv_heads + kvh) * capacity + pos;
        else
            dst_row = (static_cast<size_t>(layer * n_pages + page) * n_kv_heads + kvh) * page_size +
                      pos % page_size;
        if (which == 0)
            k[dst_row * 16 + ch] = k_new[src];
        else
            v[dst_row * 16 + ch] = v_new[src];
    }
    __syncthreads();
    if (tid == 0)
        seq_len[b] = pos + 1;
}

// Rows of one unit per compact block: 16 half-warps x kCompactRows consecutive rows each.
constexpr int kCompactRows = 8;
constexpr int kCompactBlockRows = 16 * kCompactRows;

// Each half-warp copies kCompactRows consecutive packed rows (2 KB of K and 2 KB of V,
// contiguous in the packed buffer). The positions, then (paged) their pages, then all 16
// row loads are issued before anything waits on them, so a block spends three memory round
// trips instead of one chain of dependent loads per row.
__global__ void __launch_bounds__(256) compact_kernel(
    const uint4 *__restrict__ k, const uint4 *__restrict__ v, uint4 *__restrict__ kc,
    uint4 *__restrict__ vc, const int32_t *__restrict__ sel_idx, const int32_t *__restrict__ sel_cnt,
    int32_t *__restrict__ rows_out, const int32_t *__restrict__ seq_len,
    const uint8_t *__restrict__ active, const int32_t *__restrict__ page_table, int batch,
    int n_kv_heads, int capacity, int page_size, int n_pages, int max_pages, int n_sink,
    int n_select, uint32_t *err, int n_seq_active)
{
    // (with n_seq_active > 0 the grid covers only the active sequences' units; `active` is an
    // input complete at launch, so it is read before the wait)
    const int u = launched_unit(static_cast<int>(blockIdx.x), n_seq_active, active, batch, n_kv_heads);
    if (u < 0)
        return;
    const int kvh = u % n_kv_heads;
    const int b = (u / n_kv_heads) % batch;
    const int layer = u / (n_kv_heads * batch);
    // Dependents start only once the packed rows are written (pdl_trigger_after_writes): the
    // fast step loads them before its own wait.
    pdl_wait();
    if (active && !active[b])
        return;
    const int L = min(seq_len[b], capacity);
    const int n_s = min(n_sink, L);
    const int cnt = max(0, min(sel_cnt[u], n_select));
    const int rows = n_s + cnt;
    const int comp_cap = n_sink + n_select;
    if (blockIdx.y == 0 && threadIdx.x == 0)
        rows_out[u] = rows;
    const int sub = threadIdx.x >> 4, ch = threadIdx.x & 15;
    const int r0 = blockIdx.y * kCompactBlockRows + sub * kCompactRows;
    auto copy_rows = [&](int rb) {
        int pos[kCompactRows];
#pragma unroll
        for (int j = 0; j < kCompactRows; ++j) {
            const int r = rb + j;
            pos[j] = r >= rows ? -1
                     : r < n_s ? r
                               : __ldg(sel_idx + static_cast<size_t>(u) * n_select + (r - n_s));
        }
        long long src[kCompactRows];
#pragma unroll
        for (int j = 0; j < kCompactRows; ++j) {
            const bool in = pos[j] >= 0 && pos[j] < L;
            if (page_size == 0) {
                src[j] = in ? static_cast<long long>(u) * capacity + pos[j] : -1;
            } else {
                const int page = in ? __ldg(page_table + b * max_pages + pos[j] / page_size) : -1;
                const bool good = page >= 0 && page < n_pages;
                if (in && !good && ch == 0)
                    raise_error(err, 0x1u);  // SFI_DEVERR_PAGE_RANGE: row skipped
                src[j] = (in && good) ? (static_cast<long long>(layer * n_pages + page) * n_kv_heads + kvh) *
                                                page_size + pos[j] % page_size
                                      : -1;
            }
        }
        uint4 kx[kCompactRows], vx[kCompactRows];
#pragma unroll
        for (int j = 0; j < kCompactRows; ++j) {
            if (src[j] >= 0) {
                kx[j] = __ldg(k + src[j] * 16 + ch);
                vx[j] = __ldg(v + src[j] * 16 + ch);
            }
        }
        const size_t dst0 = static_cast<size_t>(u) * comp_cap + rb;
#pragma unroll
        for (int j = 0; j < kCompactRows; ++j) {
            if (src[j] >= 0) {
                kc[(dst0 + j) * 16 + ch] = kx[j];
                vc[(dst0 + j) * 16 + ch] = vx[j];
            }
        }
    };
    if (r0 < rows)
        copy_rows(r0);
    __syncthreads();
    pdl_trigger_after_writes();
}

}  // namespace

cudaError_t launch_append(const void *k_new, const void *v_new, void *k, void *v, int32_t *seq_len,
                          const uint8_t *active, const int32_t *page_table, int n_layers, int batch,
                          int n_kv_heads, int capacity, int page_size, int n_pages, int max_pages,
                          uint32_t *err, cudaStream_t stream)
{
    const cudaError_t e = launch_pdl(
        append_kernel, dim3(batch), dim3(256), 0, stream, static_cast<const uint4 *>(k_new),
        static_cast<const uint4 *>(v_new), static_cast<uint4 *>(k), static_cast<uint4 *>(v),
        seq_len, active, page_table, n_layers, batch, n_kv_heads, capacity, page_size, n_pages,
        max_pages, err);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_compact(const void *k, const void *v, void *kc, void *vc, const int32_t *sel_idx,
                           const int32_t *sel_cnt, int32_t *rows, const int32_t *seq_len,
                           const uint8_t *active, const int32_t *page_table, int n_layers, int batch,
                           int n_kv_heads, int capacity, int page_size, int n_pages, int max_pages,
                           int n_sink, int n_select, uint32_t *err, cudaStream_t stream,
                           int n_seq_active)
{
    const int units = n_layers * (n_seq_active > 0 ? n_seq_active : batch) * n_kv_heads;
    const int comp_cap = n_sink + n_select;
    dim3 grid(units, (comp_cap + kCompactBlockRows - 1) / kCompactBlockRows);
    const cudaError_t e = launch_pdl(
        compact_kernel, grid, dim3(256), 0, stream, static_cast<const uint4 *>(k),
        static_cast<const uint4 *>(v), static_cast<uint4 *>(kc), static_cast<uint4 *>(vc), sel_idx,
        sel_cnt, rows, seq_len, active, page_table, batch, n_kv_heads, capacity, page_size, n_pages,
        max_pages, n_sink, n_select, err, n_seq_active);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace sfi
