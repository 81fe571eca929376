// api.cu -- the C ABI declared in include/gqa_attn.h: argument validation,
// per-device state (SM count, error word, registered workspace), tensor-map
// encoding, and dispatch to the kernel launchers.  No entry point allocates
// or frees device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <mutex>
#include <string.h>
#include <vector>

#include "internal.h"
#include "sm100.cuh"

namespace gqa {

// One error word per device (module-scope device memory, not an allocation),
// and where gqa_get_device_error's exchange leaves its old value.
__device__ unsigned g_err_word;
__device__ unsigned g_err_snapshot;

// Reads and clears the error word in one atomic step.
__global__ void err_exchange_kernel() { g_err_snapshot = atomicExch(&g_err_word, 0u); }

// The kernels' bounded pipeline wait on an mbarrier that nothing arrives on:
// it gives up after its limit, records the timeout in *err and returns.
__global__ void wait_limit_kernel(unsigned* err) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, err);
}

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    DeviceInfo info{};
    void* ws = nullptr;
    size_t ws_bytes = 0;
};

DeviceState g_dev[kMaxDevices];
std::mutex g_mu;
// Kernels whose dynamic shared-memory limit was raised, per device.
std::vector<const void*> g_smem_done[kMaxDevices];
EncodeTiledFn g_encode = nullptr;

}  // namespace

const DeviceInfo* device_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& st = g_dev[dev];
    if (!st.ready) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return nullptr;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return nullptr;
        st.info.device = dev;
        st.info.num_sms = sms;
        st.info.err_word = static_cast<unsigned*>(p);
        st.ready = true;
    }
    return &st.info;
}

int ensure_smem_limit(const void* kernel, int bytes) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    std::vector<const void*>& done = g_smem_done[dev];
    for (const void* k : done)
        if (k == kernel) return GQA_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess)
        return GQA_ERR_CUDA;
    done.push_back(kernel);
    return GQA_OK;
}

void current_workspace(void** ptr, size_t* bytes) {
    int dev = 0;
    *ptr = nullptr;
    *bytes = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return;
    std::lock_guard<std::mutex> lk(g_mu);
    *ptr = g_dev[dev].ws;
    *bytes = g_dev[dev].ws_bytes;
}

EncodeTiledFn encode_tiled() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return g_encode;
}

bool make_map_2d_f16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                     uint64_t row_stride, uint32_t box_rows, uint32_t box_cols) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {row_stride * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_map_3d_f16(CUtensorMap* map, const void* base, uint64_t d, uint64_t heads,
                     uint64_t rows, uint64_t head_stride, uint64_t row_stride,
                     uint32_t box_rows) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    cuuint64_t dims[3] = {d, heads, rows};
    cuuint64_t strides[2] = {head_stride, row_stride};
    cuuint32_t box[3] = {64, 1, box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_map_2d_u8(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint64_t row_stride, uint32_t box_rows, uint32_t box_cols) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {row_stride};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace gqa

using namespace gqa;

namespace {

// Every entry point takes any grouping with head size 256 or 128: Hkv KV
// heads, each shared by Hq / Hkv query heads.
bool family_ok(int Hq, int Hkv, int D) {
    return (D == kHeadDim || D == 128) && Hq >= 1 && Hq <= kMaxHeads && Hkv >= 1 &&
           Hq % Hkv == 0;
}

// One tail launch packs query_rows x (Hq / Hkv) rows into the UMMA N dimension.
bool tail_family_ok(int Hq, int Hkv, int D, int query_rows) {
    return family_ok(Hq, Hkv, D) && (long long)query_rows * (Hq / Hkv) <= kMaxTailPackedRows;
}

bool scale_ok(float s) { return isfinite(s) && s > 0.f; }

}  // namespace

namespace {

int sparse_common(const void* q, const void* kcache, const void* vcache, const float* kscale,
                  const float* vscale, bool e4m3, const int32_t* block_table,
                  const int32_t* sel_idx, const int32_t* sel_cnt, int max_sel, int num_pages,
                  int page, int ctx_len, int query_rows, int Hq, int Hkv, int D, float scale,
                  void* out, struct CUstream_st* stream) {
    if (!q || !kcache || !vcache || !block_table || !sel_idx || !sel_cnt || !out)
        return GQA_ERR_INVALID_ARG;
    if (e4m3 && (!kscale || !vscale)) return GQA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(out))
        return GQA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(block_table) | reinterpret_cast<uintptr_t>(sel_idx) |
         reinterpret_cast<uintptr_t>(sel_cnt) | reinterpret_cast<uintptr_t>(kscale) |
         reinterpret_cast<uintptr_t>(vscale)) & 3u)
        return GQA_ERR_INVALID_ARG;
    if (query_rows < 1 || ctx_len < query_rows || num_pages < 1 || max_sel < 1 ||
        !scale_ok(scale))
        return GQA_ERR_INVALID_ARG;
    if (!family_ok(Hq, Hkv, D) || Hq / Hkv > kMaxSparseGroup || !page_ok(page))
        return GQA_ERR_UNSUPPORTED;
    // Cache token rows are 32-bit indices inside the kernel.
    if ((long long)num_pages * page > 0x7fffffffLL) return GQA_ERR_UNSUPPORTED;
    if ((long long)ctx_len > (long long)num_pages * page) return GQA_ERR_INVALID_ARG;
    return sparse_launch(q, kcache, vcache, kscale, vscale, e4m3, block_table, sel_idx, sel_cnt,
                         max_sel, num_pages, page, ctx_len, query_rows, Hq, Hkv, D, scale, out,
                         stream);
}

}  // namespace

extern "C" {

int gqa_attn_prefill(const void* q, const void* k, const void* v, void* out, int Q, int KV,
                     int Hq, int Hkv, int D, float scale, struct CUstream_st* stream) {
    if (!q || !k || !v || !out) return GQA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return GQA_ERR_INVALID_ARG;
    if (Q < 1 || KV < 1 || Q > KV || !scale_ok(scale)) return GQA_ERR_INVALID_ARG;
    if (!family_ok(Hq, Hkv, D)) return GQA_ERR_UNSUPPORTED;
    if ((long long)Q * Hq > 0x7fffffffLL - 256) return GQA_ERR_INVALID_ARG;
    return prefill_launch(q, k, v, nullptr, nullptr, out, Q, KV, Hq, Hkv, D, scale, stream);
}

int gqa_attn_prefill_e4m3(const void* q, const uint8_t* k, const uint8_t* v, const float* kscale,
                          const float* vscale, void* out, int Q, int KV, int Hq, int Hkv, int D,
                          float scale, struct CUstream_st* stream) {
    if (!q || !k || !v || !kscale || !vscale || !out) return GQA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return GQA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(kscale) | reinterpret_cast<uintptr_t>(vscale)) & 3u)
        return GQA_ERR_INVALID_ARG;
    if (Q < 1 || KV < 1 || Q > KV || !scale_ok(scale)) return GQA_ERR_INVALID_ARG;
    if (!family_ok(Hq, Hkv, D)) return GQA_ERR_UNSUPPORTED;
    if ((long long)Q * Hq > 0x7fffffffLL - 256) return GQA_ERR_INVALID_ARG;
    return prefill_launch(q, k, v, kscale, vscale, out, Q, KV, Hq, Hkv, D, scale, stream);
}

int gqa_attn_paged_e4m3(const void* q, const uint8_t* kcache, const uint8_t* vcache,
                        const float* kscale, const float* vscale, const int32_t* block_table,
                        int num_pages, int page, int ctx_len, int query_rows, int Hq, int Hkv,
                        int D, float scale, void* out, struct CUstream_st* stream) {
    if (!q || !kcache || !vcache || !kscale || !vscale || !block_table || !out)
        return GQA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(out))
        return GQA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(kscale) | reinterpret_cast<uintptr_t>(vscale) |
         reinterpret_cast<uintptr_t>(block_table)) & 3u)
        return GQA_ERR_INVALID_ARG;
    if (query_rows < 1 || ctx_len < query_rows || num_pages < 1 || !scale_ok(scale))
        return GQA_ERR_INVALID_ARG;
    if (!tail_family_ok(Hq, Hkv, D, query_rows) || !page_ok(page)) return GQA_ERR_UNSUPPORTED;
    if ((long long)ctx_len > (long long)num_pages * page) return GQA_ERR_INVALID_ARG;
    return paged_e4m3_launch(q, kcache, vcache, kscale, vscale, block_table, num_pages, page,
                             ctx_len, nullptr, query_rows, Hq, Hkv, D, scale, out, stream);
}

int gqa_attn_paged_e4m3_batch(const void* q, const uint8_t* kcache, const uint8_t* vcache,
                              const float* kscale, const float* vscale,
                              const int32_t* block_tables, int table_stride, int num_pages,
                              int page, const int32_t* ctx_lens_dev, int max_ctx_len, int batch,
                              int query_rows, int Hq, int Hkv, int D, float scale, void* out,
                              struct CUstream_st* stream) {
    if (!q || !kcache || !vcache || !kscale || !vscale || !block_tables || !ctx_lens_dev || !out)
        return GQA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(out))
        return GQA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(kscale) | reinterpret_cast<uintptr_t>(vscale) |
         reinterpret_cast<uintptr_t>(block_tables) | reinterpret_cast<uintptr_t>(ctx_lens_dev)) &
        3u)
        return GQA_ERR_INVALID_ARG;
    if (query_rows < 1 || max_ctx_len < query_rows || num_pages < 1 || batch < 1 ||
        !scale_ok(scale))
        return GQA_ERR_INVALID_ARG;
    if (!tail_family_ok(Hq, Hkv, D, query_rows) || !page_ok(page) || batch > kMaxTailBatch)
        return GQA_ERR_UNSUPPORTED;
    if ((long long)max_ctx_len > (long long)num_pages * page) return GQA_ERR_INVALID_ARG;
    if ((long long)table_stride * page < (long long)max_ctx_len) return GQA_ERR_INVALID_ARG;
    return paged_e4m3_batch_launch(q, kcache, vcache, kscale, vscale, block_tables, table_stride,
                                   num_pages, page, ctx_lens_dev, max_ctx_len, batch, query_rows,
                                   Hq, Hkv, D, scale, out, stream);
}

int gqa_attn_paged_e4m3_devctx(const void* q, const uint8_t* kcache, const uint8_t* vcache,
                               const float* kscale, const float* vscale,
                               const int32_t* block_table, int num_pages, int page,
                               const int32_t* ctx_len_dev, int max_ctx_len, int query_rows,
                               int Hq, int Hkv, int D, float scale, void* out,
                               struct CUstream_st* stream) {
    if (!q || !kcache || !vcache || !kscale || !vscale || !block_table || !ctx_len_dev || !out)
        return GQA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(out))
        return GQA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(kscale) | reinterpret_cast<uintptr_t>(vscale) |
         reinterpret_cast<uintptr_t>(block_table) | reinterpret_cast<uintptr_t>(ctx_len_dev)) &
        3u)
        return GQA_ERR_INVALID_ARG;
    if (query_rows < 1 || max_ctx_len < query_rows || num_pages < 1 || !scale_ok(scale))
        return GQA_ERR_INVALID_ARG;
    if (!tail_family_ok(Hq, Hkv, D, query_rows) || !page_ok(page)) return GQA_ERR_UNSUPPORTED;
    if ((long long)max_ctx_len > (long long)num_pages * page) return GQA_ERR_INVALID_ARG;
    return paged_e4m3_launch(q, kcache, vcache, kscale, vscale, block_table, num_pages, page,
                             max_ctx_len, ctx_len_dev, query_rows, Hq, Hkv, D, scale, out,
                             stream);
}

int gqa_attn_paged_e4m3_noalloc(const void* q, const uint8_t* kcache, const uint8_t* vcache,
                                const float* kscale, const float* vscale,
                                const int32_t* block_table, int num_pages, int page, int ctx_len,
                                int query_rows, int Hq, int Hkv, int D, float scale, void* out,
                                struct CUstream_st* stream) {
    if (!q || !kcache || !vcache || !kscale || !vscale || !block_table || !out)
        return GQA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(out))
        return GQA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(kscale) | reinterpret_cast<uintptr_t>(vscale) |
         reinterpret_cast<uintptr_t>(block_table)) & 3u)
        return GQA_ERR_INVALID_ARG;
    if (query_rows < 1 || ctx_len < query_rows || num_pages < 1 || !scale_ok(scale))
        return GQA_ERR_INVALID_ARG;
    if (!tail_family_ok(Hq, Hkv, D, query_rows) || !page_ok(page)) return GQA_ERR_UNSUPPORTED;
    if ((long long)ctx_len > (long long)num_pages * page) return GQA_ERR_INVALID_ARG;
    return paged_e4m3_noalloc_launch(q, kcache, vcache, kscale, vscale, block_table, num_pages,
                                     page, ctx_len, query_rows, Hq, Hkv, D, scale, out, stream);
}

int gqa_attn_sparse_blocks(const void* q, const void* kcache, const void* vcache,
                           const int32_t* block_table, const int32_t* sel_idx,
                           const int32_t* sel_cnt, int max_sel, int num_pages, int page,
                           int ctx_len, int query_rows, int Hq, int Hkv, int D, float scale,
                           void* out, struct CUstream_st* stream) {
    return sparse_common(q, kcache, vcache, nullptr, nullptr, false, block_table, sel_idx,
                         sel_cnt, max_sel, num_pages, page, ctx_len, query_rows, Hq, Hkv, D,
                         scale, out, stream);
}

int gqa_attn_sparse_blocks_e4m3(const void* q, const uint8_t* kcache, const uint8_t* vcache,
                                const float* kscale, const float* vscale,
                                const int32_t* block_table, const int32_t* sel_idx,
                                const int32_t* sel_cnt, int max_sel, int num_pages, int page,
                                int ctx_len, int query_rows, int Hq, int Hkv, int D, float scale,
                                void* out, struct CUstream_st* stream) {
    return sparse_common(q, kcache, vcache, kscale, vscale, true, block_table, sel_idx, sel_cnt,
                         max_sel, num_pages, page, ctx_len, query_rows, Hq, Hkv, D, scale, out,
                         stream);
}

size_t gqa_workspace_bytes(int kind, int query_rows, int ctx_or_kv, int Hq, int D) {
    if ((D != kHeadDim && D != 128) || query_rows < 1 || ctx_or_kv < 1) return 0;
    if (Hq < 1 || Hq > kMaxHeads) return 0;
    const DeviceInfo* di = device_info();
    if (!di) return 0;
    // The tail's partials are sized for query_rows x Hq packed rows, enough
    // for any number of KV heads (one launch takes query_rows x Hq / Hkv).
    if (kind == GQA_KIND_PAGED_E4M3_BATCH) {   // ctx_or_kv = number of sequences
        if (query_rows > kMaxTailPackedRows || ctx_or_kv > kMaxTailBatch) return 0;
        return paged_e4m3_batch_workspace_bytes(query_rows * Hq, ctx_or_kv, di->num_sms, D);
    }
    if (ctx_or_kv < query_rows) return 0;
    switch (kind) {
        case GQA_KIND_PREFILL:
            return prefill_workspace_bytes(query_rows, ctx_or_kv, di->num_sms);
        case GQA_KIND_PAGED_E4M3:
            if (query_rows > kMaxTailPackedRows) return 0;
            return paged_e4m3_workspace_bytes(query_rows * Hq, ctx_or_kv, di->num_sms, D);
        case GQA_KIND_SPARSE:
            return kWorkspaceCounterBytes;
        default:
            return 0;
    }
}

int gqa_set_workspace(int device, void* ptr, size_t bytes) {
    if (device < 0 || device >= 64) return GQA_ERR_INVALID_ARG;
    if (ptr && ((reinterpret_cast<uintptr_t>(ptr) & 255u) || bytes < kWorkspaceCounterBytes))
        return GQA_ERR_INVALID_ARG;
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return GQA_ERR_CUDA;
    if (ptr) {
        if (cudaSetDevice(device) != cudaSuccess) return GQA_ERR_CUDA;
        cudaError_t e = cudaMemset(ptr, 0, kWorkspaceCounterBytes);
        cudaSetDevice(prev);
        if (e != cudaSuccess) return GQA_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    g_dev[device].ws = ptr;
    g_dev[device].ws_bytes = ptr ? bytes : 0;
    return GQA_OK;
}

int gqa_get_device_error(struct CUstream_st* stream) {
    const DeviceInfo* di = device_info();
    if (!di) return -1;
    // After the stream's earlier work, swap the word for 0 on the device (a
    // bit set concurrently by a kernel on another stream is never lost), then
    // read the old value back.
    err_exchange_kernel<<<1, 1, 0, stream>>>();
    if (cudaGetLastError() != cudaSuccess) return -1;
    unsigned v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_err_snapshot, sizeof v, 0, cudaMemcpyDeviceToHost,
                                  stream) != cudaSuccess)
        return -1;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return -1;
    return (int)v;
}

int gqa_check_wait_limit(struct CUstream_st* stream) {
    const DeviceInfo* di = device_info();
    if (!di) return GQA_ERR_CUDA;
    wait_limit_kernel<<<1, 32, 0, stream>>>(di->err_word);
    return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

int gqa_prefill_sm_pairs(void) { return prefill_resident_pairs(); }

const char* gqa_status_string(int status) {
    switch (status) {
        case GQA_OK: return "GQA_OK";
        case GQA_ERR_INVALID_ARG: return "GQA_ERR_INVALID_ARG";
        case GQA_ERR_UNSUPPORTED: return "GQA_ERR_UNSUPPORTED";
        case GQA_ERR_WORKSPACE: return "GQA_ERR_WORKSPACE";
        case GQA_ERR_CUDA: return "GQA_ERR_CUDA";
        default: return "GQA_UNKNOWN_STATUS";
    }
}

}  // extern "C"
