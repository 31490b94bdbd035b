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

__global__ void __launch_bounds__(256) compact_kernel(
    const uint4 *__restrict__ k, const uint4 *__restrict__ v, uint4 *__restrict__ kc,
    uint4 *__restrict__ vc, const int32_t *__restrict__ sel_idx, const int32_t *__restrict__ sel_cnt,
    int32_t *__restrict__ rows_out, const int32_t *__restrict__ seq_len,
    const uint8_t *__restrict__ active, const int32_t *__restrict__ page_table, int batch,
    int n_kv_heads, int capacity, int page_size, int n_pages, int max_pages, int n_sink,
    int n_select, uint32_t *err)
{
    const int u = blockIdx.x;
    const int kvh = u % n_kv_heads;
    const int b = (u / n_kv_heads) % batch;
    const int layer = u / (n_kv_heads * batch);
    pdl_trigger();
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
    for (int r = blockIdx.y * 16 + sub; r < rows; r += gridDim.y * 16) {
        const int pos = r < n_s ? r : __ldg(sel_idx + static_cast<size_t>(u) * n_select + (r - n_s));
        if (pos < 0 || pos >= L)
            continue;
        size_t src_row;
        if (page_size == 0) {
            src_row = static_cast<size_t>(u) * capacity + pos;
        } else {
            const int page = __ldg(page_table + b * max_pages + pos / page_size);
            if (page < 0 || page >= n_pages) {
                if (ch == 0)
                    raise_error(err, 0x1u);
                continue;
            }
            src_row = (static_cast<size_t>(layer * n_pages + page) * n_kv_heads + kvh) * page_size +
                      pos % page_size;
        }
        const size_t dst_row = static_cast<size_t>(u) * comp_cap + r;
        kc[dst_row * 16 + ch] = __ldg(k + src_row * 16 + ch);
        vc[dst_row * 16 + ch] = __ldg(v + src_row * 16 + ch);
    }
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
                           int n_sink, int n_select, uint32_t *err, cudaStream_t stream)
{
    const int units = n_layers * batch * n_kv_heads;
    const int comp_cap = n_sink + n_select;
    dim3 grid(units, (comp_cap + 127) / 128);
    const cudaError_t e = launch_pdl(
        compact_kernel, grid, dim3(256), 0, stream, static_cast<const uint4 *>(k),
        static_cast<const uint4 *>(v), static_cast<uint4 *>(kc), static_cast<uint4 *>(vc), sel_idx,
        sel_cnt, rows, seq_len, active, page_table, batch, n_kv_heads, capacity, page_size, n_pages,
        max_pages, n_sink, n_select, err);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace sfi
