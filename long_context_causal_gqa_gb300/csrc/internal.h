// internal.h -- host-side declarations shared by the library's translation
// units (not part of the public C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/gqa_attn.h"

namespace gqa {

constexpr int kHq = 6;
constexpr int kHkv = 1;
constexpr int kHeadDim = 256;
constexpr int kMaxHeads = 64;          // query heads accepted by the prefill and the E4M3 tail
constexpr int kMaxTailPackedRows = 48; // query rows x query heads per KV head in one tail launch
constexpr int kMaxSparseGroup = 16;    // query heads per KV head in one sparse launch
constexpr int kPage = 16;   // the pages' page size; any power of two in [8, 256] is accepted

// Page sizes the paged kernels take: a power of two in [8, 256] (so that a
// 4-token block never straddles a page and a 128-key tile is whole pages or a
// slice of one).
inline bool page_ok(int page) { return page >= 8 && page <= 256 && (page & (page - 1)) == 0; }

// Most sequences one batched tail launch takes (its merge reads at most 1024
// split partials per packed row).
constexpr int kMaxTailBatch = 1024;

struct DeviceInfo {
    int device;
    int num_sms;
    unsigned* err_word;  // device address of this device's error word
};

// Per-device facts, looked up once; returns nullptr on a CUDA error.
const DeviceInfo* device_info();

// Workspace registered for the current device (ptr may be null).
void current_workspace(void** ptr, size_t* bytes);

// cuTensorMapEncodeTiled, fetched through the runtime's driver entry point.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled();

// 2D fp16 tensor [rows, cols], rows row_stride elements apart (a multiple of
// 8), with a box of [box_rows, box_cols] (box_cols * 2 bytes <= 128), 128-byte
// swizzle, zero fill out of bounds.
bool make_map_2d_f16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                     uint64_t row_stride, uint32_t box_rows, uint32_t box_cols);

// 3D fp16 tensor (d, heads, rows) with heads head_stride bytes apart and rows
// row_stride bytes apart (multiples of 16), a box of 64 d x 1 head x box_rows
// rows, 128-byte swizzle, zero fill out of bounds.
bool make_map_3d_f16(CUtensorMap* map, const void* base, uint64_t d, uint64_t heads,
                     uint64_t rows, uint64_t head_stride, uint64_t row_stride,
                     uint32_t box_rows);

// 2D uint8 tensor [rows, cols], rows row_stride bytes apart (a multiple of
// 16), with a box of [box_rows, box_cols] (box_cols <= 128), 128-byte swizzle.
bool make_map_2d_u8(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint64_t row_stride, uint32_t box_rows, uint32_t box_cols);

// Exact unsigned division by a divisor fixed per launch, for dividends below
// 2^31: the multiply-high method of Granlund and Montgomery ("Division by
// invariant integers using multiplication", 1994, section 4), with
// l = ceil(log2 d) and mul = floor(2^32 (2^l - d) / d) + 1.
struct FastDiv {
    uint32_t mul;
    int shift;
    int d;
    __host__ __device__ int div(int n) const {
#ifdef __CUDA_ARCH__
        return (int)((__umulhi(mul, (uint32_t)n) + (uint32_t)n) >> shift);
#else
        return n / d;
#endif
    }
};

inline FastDiv make_fastdiv(int d) {
    FastDiv f;
    f.d = d;
    int l = 0;
    while ((1LL << l) < d) ++l;
    f.shift = l;
    f.mul = (uint32_t)((((1ULL << l) - (unsigned long long)d) << 32) / (unsigned long long)d + 1);
    return f;
}

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device); thread-safe.  GQA_OK or GQA_ERR_CUDA.
int ensure_smem_limit(const void* kernel, int bytes);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launchers (one per kernel family).  Arguments are validated by the caller.
// Dh: head size, 256 or 128.
// kscale / vscale: null for fp16 k / v; device pointers to one fp32 each when
// k / v hold E4M3 codes.
int prefill_launch(const void* q, const void* k, const void* v, const float* kscale,
                   const float* vscale, void* out, int Q, int KV, int Hq, int Hkv, int Dh,
                   float scale, cudaStream_t stream);
size_t prefill_workspace_bytes(int Q, int KV, int num_sms);
int prefill_resident_pairs();   // co-resident two-CTA clusters of the prefill kernel

int paged_e4m3_launch(const void* q, const uint8_t* kcache, const uint8_t* vcache,
                      const float* kscale, const float* vscale, const int32_t* block_table,
                      int num_pages, int page, int ctx_len, const int* ctx_dev, int R,
                      int Hq, int Hkv, int Dh, float scale, void* out, cudaStream_t stream);
// nq = packed rows of one launch (at most query_rows * Hq); Dh = head size.
size_t paged_e4m3_workspace_bytes(int nq, int ctx_len, int num_sms, int Dh);
int paged_e4m3_batch_launch(const void* q, const uint8_t* kcache, const uint8_t* vcache,
                            const float* kscale, const float* vscale,
                            const int32_t* block_tables, int table_stride, int num_pages,
                            int page, const int* ctx_lens_dev, int max_ctx_len, int batch,
                            int R, int Hq, int Hkv, int Dh, float scale, void* out,
                            cudaStream_t stream);
size_t paged_e4m3_batch_workspace_bytes(int nq, int batch, int num_sms, int Dh);

// Same as paged_e4m3_launch, with the split partials in a static device array.
int paged_e4m3_noalloc_launch(const void* q, const uint8_t* kcache, const uint8_t* vcache,
                              const float* kscale, const float* vscale,
                              const int32_t* block_table, int num_pages, int page, int ctx_len,
                              int R, int Hq, int Hkv, int Dh, float scale, void* out,
                              cudaStream_t stream);

// kcache / vcache: fp16 elements, or E4M3 codes with kscale / vscale (device
// pointers to one fp32 each) when e4m3 is set.
int sparse_launch(const void* q, const void* kcache, const void* vcache, const float* kscale,
                  const float* vscale, bool e4m3, const int32_t* block_table,
                  const int32_t* sel_idx, const int32_t* sel_cnt, int max_sel, int num_pages,
                  int page, int ctx_len, int rows, int Hq, int Hkv, int Dh, float scale,
                  void* out, cudaStream_t stream);

// Bytes at the start of every workspace reserved for merge counters.
constexpr size_t kWorkspaceCounterBytes = 4096;

}  // namespace gqa
