/*
 * gqa_attn.h -- C ABI of libgqa_attn.so: causal grouped-query attention on
 * NVIDIA GB300 (sm_103a).
 *
 *   out[i, h, :] = softmax_j( scale * q[i, h, :] . k[j, g, :] )  v[j, g, :]
 *
 * over the keys j that query row i may see, with g = h / (Hq / Hkv) the KV
 * head shared by a group of query heads.  Query rows are bottom-right
 * aligned: with R query rows and a context of N keys, row i sits at absolute
 * position N - R + i and sees keys 0 .. N - R + i.
 *
 * Sources (web pages, by title and section):
 *   [P1] "[Kernel][SM70] Default long-prefill GQA architecture", Purpose:
 *        causal FP16 prefill, Q=8000, KV=40000..128000, Hq=6, Hkv=1, D=256,
 *        scale 1/16; Test Result: FP16 envelope max abs <= 1e-3, rel L2 <= 1e-2.
 *   [P2] "[Perf] Ship the qualified SM70 long-context layout and drop its
 *        context fences", What / Changes: grouped E4M3 FP32 long-context
 *        operator, capacity 262144, verifier tails of 1..8 query rows.
 *   [P3] "[Kernel][SM70] Repair #378 on latest main", Changes: per-row
 *        selected four-token KV blocks over a page-16 cache whose block table
 *        is in physical-page units; positions clamped to the row.
 *
 * Conventions shared by every entry point
 *   - Head sizes and groupings: D = 256 or 128 for every entry point; Hkv KV
 *     heads, each shared by Hq / Hkv query heads (Hkv divides Hq, Hq <= 64).
 *     The pages' family is Hq = 6, Hkv = 1, D = 256; with Hkv > 1 the
 *     prefill gives every query head its own tiles in one launch and the
 *     E4M3 tail and sparse entry points run one launch per KV head, with
 *     per-entry limits below.  Anything else returns GQA_ERR_UNSUPPORTED.
 *     scale must be finite and > 0.
 *   - All tensor pointers are DEVICE pointers, contiguous, 16-byte aligned,
 *     owned by the caller.  fp16 means IEEE binary16.
 *   - q / out are [rows, Hq, D] fp16; out is fully overwritten.
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream) and
 *     never allocate or free memory.  Work that needs scratch space (split
 *     partials, merge counters) uses the workspace registered with
 *     gqa_set_workspace for the current device; calls that share one
 *     workspace must not overlap on the GPU (issue them on one stream).
 *   - Results are bitwise reproducible from run to run and under CUDA-graph
 *     replay: the work partition depends only on the shape and the device's
 *     SM count, and every reduction has a fixed order.
 *   - The first call of each entry point on a device loads its kernels and
 *     sets their shared-memory limits; make it before capturing a graph.
 *   - Return value: a gqa_status.  Argument errors are detected on the host
 *     before anything is launched.  Errors found on the device (out-of-range
 *     block ids, a pipeline wait that timed out) set a per-device error word
 *     read by gqa_get_device_error; the kernel masks the offending input and
 *     carries on (or returns) instead of trapping.
 */
#ifndef GQA_ATTN_H
#define GQA_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t */

typedef enum {
    GQA_OK = 0,
    GQA_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, bad size, rows > context, bad scale */
    GQA_ERR_UNSUPPORTED = 2,   /* D not 128 or 256, Hkv not dividing Hq,
                                  Hq > 64, page not a power of
                                  two in [8, 256], query_rows * Hq / Hkv > 48 (E4M3 tail),
                                  Hq / Hkv > 16 (sparse) */
    GQA_ERR_WORKSPACE = 3,     /* no workspace registered, or it is too small */
    GQA_ERR_CUDA = 4           /* a CUDA runtime call or kernel launch failed */
} gqa_status;

/* Bits of the device error word (gqa_get_device_error). */
#define GQA_DEVERR_WAIT_TIMEOUT 0x1u  /* a pipeline wait exceeded its limit; output invalid */
#define GQA_DEVERR_BAD_BLOCK_ID 0x2u  /* sel_idx held an id < 0 or past the row's own block */
#define GQA_DEVERR_BAD_PAGE_ID  0x4u  /* a block-table entry was < 0 or >= num_pages */
#define GQA_DEVERR_BAD_CTX_LEN  0x8u  /* a device-side ctx_len was < query_rows or > max_ctx_len */
#define GQA_DEVERR_DUP_BLOCK_ID 0x10u /* sel_idx held an id an earlier position of its row holds */

/* Dense causal prefill [P1, Purpose].
 *   q   [Q, Hq, D]  fp16     k, v [KV, Hkv, D] fp16     out [Q, Hq, D] fp16
 *   1 <= Q <= KV.  Row i sees keys 0 .. KV - Q + i.
 * With Hkv = 1 the Q x Hq rows are packed into 128-row tiles in one launch;
 * with Hkv > 1 every query head has its own row tiles (one row per position)
 * in the same launch, read in place through strided views.  FP32
 * accumulation; P is rounded to fp16 before the P.V product; the output
 * is rounded to nearest fp16.  Long problems are split over all SMs; the
 * split partials live in the registered workspace
 * (gqa_workspace_bytes(GQA_KIND_PREFILL, Q, KV, Hq, D) bytes). */
int gqa_attn_prefill(const void* q, const void* k, const void* v, void* out, int Q, int KV,
                     int Hq, int Hkv, int D, float scale, struct CUstream_st* stream);

/* Dense causal prefill over an FP8-E4M3 K/V cache: the E4M3 storage of
 * [P2, What] applied to the dense workload of [P1, Purpose].  Same arguments,
 * layouts and result as gqa_attn_prefill, except:
 *   k, v          [KV, Hkv, D] uint8 E4M3 codes (OCP e4m3fn: bias 7, 0x7F /
 *                 0xFF NaN, max 448); real value = decode(byte) * scale; no
 *                 code may be the NaN code
 *   kscale/vscale DEVICE pointers to one fp32 each, 4-byte aligned
 *                 (graph-capturable)
 * Each CTA's tensor-memory copies bring the codes into shared memory, where
 * two converter warps write them as fp16 (exact: every E4M3 value is an fp16
 * value) into the slots the fp16 UMMAs read; the K scale joins the score
 * scale and the V scale multiplies the output.  Half the K/V bytes of the
 * fp16 prefill; the workspace is the same (GQA_KIND_PREFILL). */
int gqa_attn_prefill_e4m3(const void* q, const uint8_t* k, const uint8_t* v, const float* kscale,
                          const float* vscale, void* out, int Q, int KV, int Hq, int Hkv, int D,
                          float scale, struct CUstream_st* stream);

/* Paged FP8-E4M3 verifier tail [P2, What / Changes].
 *   q            [query_rows, Hq, D] fp16, 1 <= query_rows, query_rows * Hq / Hkv
 *                <= 48 (one launch per KV head packs its query heads x rows;
 *                the pages' tails are 1..8 rows of 6 heads)
 *   kcache/vcache [num_pages, page, Hkv, D] uint8 E4M3 codes (OCP e4m3fn:
 *                bias 7, 0x7F/0xFF NaN, max 448); real value = decode(byte) * scale
 *   kscale/vscale DEVICE pointers to one fp32 each (graph-capturable)
 *   block_table  [ceil(ctx_len / page)] int32 physical page ids, each in
 *                [0, num_pages); entries outside it are clamped to page 0 and
 *                flag GQA_DEVERR_BAD_PAGE_ID
 *   page: tokens per cache page, a power of two in [8, 256] (the pages use 16);
 *   query_rows <= ctx_len <= num_pages * page.
 * Tail row r sits at position ctx_len - query_rows + r.  The key range is
 * split over all SMs; each split's (O, m, l) partial goes to the workspace
 * and a second kernel on the same stream merges them in a fixed order. */
int gqa_attn_paged_e4m3(const void* q, const uint8_t* kcache, const uint8_t* vcache,
                        const float* kscale, const float* vscale, const int32_t* block_table,
                        int num_pages, int page, int ctx_len, int query_rows, int Hq, int Hkv,
                        int D, float scale, void* out, struct CUstream_st* stream);

/* Paged FP8-E4M3 verifier tail whose context length is read on the device
 * when the kernels run ([P2] Changes: the tail CUDA graph is captured once for
 * a bound and replayed while the context grows).  Same arguments, layouts and
 * result as gqa_attn_paged_e4m3, except:
 *   ctx_len_dev  device pointer to one int32, the context length used by this
 *                launch (and by every replay of a graph that captured it);
 *                4-byte aligned.
 *   max_ctx_len  host bound: query_rows <= max_ctx_len <= num_pages * page.
 *                The grid, the workspace size (gqa_workspace_bytes with
 *                ctx_or_kv = max_ctx_len) and the part of block_table that may
 *                be read ([ceil(max_ctx_len / page)] entries) follow it.
 * A device value below query_rows or above max_ctx_len is clamped into that
 * range and flags GQA_DEVERR_BAD_CTX_LEN.  Splits that the actual context
 * leaves without keys publish empty partials, so the result equals
 * gqa_attn_paged_e4m3 at the same context up to the order of the split merge
 * (the split boundaries depend on max_ctx_len only through the SM count). */
int gqa_attn_paged_e4m3_devctx(const void* q, const uint8_t* kcache, const uint8_t* vcache,
                               const float* kscale, const float* vscale,
                               const int32_t* block_table, int num_pages, int page,
                               const int32_t* ctx_len_dev, int max_ctx_len, int query_rows,
                               int Hq, int Hkv, int D, float scale, void* out,
                               struct CUstream_st* stream);

/* Several sequences' E4M3 verifier tails in one launch ([P2] Changes; a
 * serving step verifies a batch of sequences of different lengths): the
 * batched, variable-length form of gqa_attn_paged_e4m3_devctx.  All
 * sequences share one cache (kcache/vcache, kscale/vscale, page) and
 * query_rows; per sequence b:
 *   q[b], out[b]        q/out [batch, query_rows, Hq, D] fp16
 *   block_tables[b]     [batch, table_stride] int32 physical page ids;
 *                       table_stride * page >= max_ctx_len
 *   ctx_lens_dev[b]     device int32 [batch], read when the kernels run (so a
 *                       captured graph replays as the contexts grow); each is
 *                       clamped into [query_rows, max_ctx_len] and flags
 *                       GQA_DEVERR_BAD_CTX_LEN if it was outside.
 * 1 <= batch <= 1024.  The grid has max(SM count, batch) splits, divided
 * between the sequences in proportion to their 128-key tile counts (at least
 * one each) on the device; each split's partial goes to the workspace
 * (gqa_workspace_bytes(GQA_KIND_PAGED_E4M3_BATCH, query_rows, batch, ...))
 * and a second kernel merges every sequence's splits in a fixed order. */
int gqa_attn_paged_e4m3_batch(const void* q, const uint8_t* kcache, const uint8_t* vcache,
                              const float* kscale, const float* vscale,
                              const int32_t* block_tables, int table_stride, int num_pages,
                              int page, const int32_t* ctx_lens_dev, int max_ctx_len, int batch,
                              int query_rows, int Hq, int Hkv, int D, float scale, void* out,
                              struct CUstream_st* stream);

/* Paged FP8-E4M3 verifier tail that allocates nothing (no counterpart in the
 * pages; an addition of this library).  Some callers cannot call cudaMalloc:
 * engines whose pooling allocator owns all device memory and must not see
 * foreign allocations, latency-critical serving loops in which cudaMalloc's
 * implicit device synchronisation is not acceptable, and plugin code that has
 * no access to the process's allocator.  This entry point takes the same
 * arguments, layouts and error codes as gqa_attn_paged_e4m3 and computes the
 * same result (bitwise equal on devices with at most 160 SMs), but needs no
 * registered workspace: its split partials live in a static device array
 * inside the library, at most 160 splits x 48 packed rows x 258 floats
 * (about 7.9 MB), which every GPU that loads the library holds until the
 * process exits.  It never calls cudaMalloc, cudaFree or any allocating
 * routine.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - All calls on a device share the one array, which keeps the last call's
 *     contents.  Nothing in it has to start at zero: a call writes every
 *     partial it reads.  Calls that overlap on the GPU (e.g. on two streams
 *     without ordering) race on the array and give wrong results.
 *   - query_rows * Hq / Hkv > 48 returns GQA_ERR_UNSUPPORTED; a shape whose
 *     partials would not fit the array returns GQA_ERR_WORKSPACE. */
int gqa_attn_paged_e4m3_noalloc(const void* q, const uint8_t* kcache, const uint8_t* vcache,
                                const float* kscale, const float* vscale,
                                const int32_t* block_table, int num_pages, int page,
                                int ctx_len, int query_rows, int Hq, int Hkv, int D,
                                float scale, void* out, struct CUstream_st* stream);

/* Selected-block sparse paged prefill [P3, Changes].
 *   q            [query_rows, Hq, D] fp16
 *   kcache/vcache [num_pages, page, Hkv, D] fp16, page a power of two in
 *                [8, 256] (the pages use 16)
 *   block_table  [ceil(ctx_len / page)] int32 physical page ids
 *   sel_idx      [query_rows, max_sel] int32 logical 4-token block ids b
 *                (tokens 4b .. 4b+3); sel_cnt [query_rows] int32, 0..max_sel
 * Row i (position p = ctx_len - query_rows + i) attends the tokens of its
 * first sel_cnt[i] selected blocks that are <= p; the row's own block is
 * clamped to p.  Selection has set semantics ([P3] Changes: stale or padded
 * entries are masked, not attended): an id that an earlier position of the
 * row already holds selects nothing more and flags GQA_DEVERR_DUP_BLOCK_ID;
 * ids < 0 or > p / 4 select nothing and flag GQA_DEVERR_BAD_BLOCK_ID.  The
 * order of a row's ids changes the result only within rounding.  A row that
 * selects no visible token gets a zero output.  The selection is shared by all heads of the row;
 * Hq / Hkv <= 16 (the query heads of one KV head are the N columns of one
 * launch; Hkv > 1 runs one launch per KV head).  num_pages * page must be
 * below 2^31 (GQA_ERR_UNSUPPORTED otherwise).  Needs no workspace. */
int gqa_attn_sparse_blocks(const void* q, const void* kcache, const void* vcache,
                           const int32_t* block_table, const int32_t* sel_idx,
                           const int32_t* sel_cnt, int max_sel, int num_pages, int page,
                           int ctx_len, int query_rows, int Hq, int Hkv, int D, float scale,
                           void* out, struct CUstream_st* stream);

/* Selected-block sparse paged prefill over an FP8-E4M3 page cache: the E4M3
 * storage of [P2, What] applied to the [P3, Changes] workload.  Same
 * arguments, selection semantics and result as gqa_attn_sparse_blocks,
 * except:
 *   kcache/vcache [num_pages, page, Hkv, D] uint8 E4M3 codes (OCP e4m3fn),
 *                real value = decode(byte) * scale
 *   kscale/vscale DEVICE pointers to one fp32 each, 4-byte aligned
 * The codes feed the FP8 tensor cores as they are; Q (one scale per head)
 * and the softmax weights P enter those products as three-term E4M3
 * expansions (at least fp16's 11 significant bits); the K scale multiplies
 * the scores and the V scale the output.  A selected token's code bytes must
 * not be the E4M3 NaN code (0x7F / 0xFF).  Needs no workspace. */
int gqa_attn_sparse_blocks_e4m3(const void* q, const uint8_t* kcache, const uint8_t* vcache,
                                const float* kscale, const float* vscale,
                                const int32_t* block_table, const int32_t* sel_idx,
                                const int32_t* sel_cnt, int max_sel, int num_pages, int page,
                                int ctx_len, int query_rows, int Hq, int Hkv, int D, float scale,
                                void* out, struct CUstream_st* stream);

/* Workspace kinds for gqa_workspace_bytes. */
#define GQA_KIND_PREFILL 0
#define GQA_KIND_PAGED_E4M3 1
#define GQA_KIND_SPARSE 2
#define GQA_KIND_PAGED_E4M3_BATCH 3   /* ctx_or_kv = number of sequences */

/* Bytes of workspace an entry point of `kind` needs for the given shape on
 * the current device (query_rows = Q or the tail/row count, ctx_or_kv = KV or
 * ctx_len).  The size holds for any Hkv dividing Hq.  Returns 0 for
 * unsupported arguments. */
size_t gqa_workspace_bytes(int kind, int query_rows, int ctx_or_kv, int Hq, int D);

/* Register caller-owned device memory as the workspace of `device`
 * (ptr 256-byte aligned, or NULL to unregister).  The library keeps the
 * pointer and never frees it.  Registration zeroes the small counter area at
 * the start of the workspace (a synchronous cudaMemset); kernels leave those
 * counters at zero when they finish.  After a device error
 * (gqa_get_device_error != 0) register the workspace again. */
int gqa_set_workspace(int device, void* ptr, size_t bytes);

/* After the work already queued on `stream`, read and clear the current
 * device's error word in one atomic step (a one-thread kernel on `stream`),
 * then synchronise `stream` and return it (GQA_DEVERR_* bits; 0 = no
 * device-side error since the last read).  Returns -1 if the CUDA calls
 * themselves failed. */
int gqa_get_device_error(struct CUstream_st* stream);

/* Diagnostic (an addition of this library): queues on `stream` a one-warp
 * kernel that runs the bounded wait every pipeline barrier of the library's
 * kernels uses, on an mbarrier that nothing ever arrives on.  After the
 * wait's limit (about 2 s) it gives up, sets GQA_DEVERR_WAIT_TIMEOUT in the
 * device error word and the kernel returns, so the context stays usable: a
 * caller can check that a stalled pipeline reports an error instead of
 * hanging.  Read the result with gqa_get_device_error.  Returns GQA_OK once
 * queued, GQA_ERR_CUDA if the launch failed. */
int gqa_check_wait_limit(struct CUstream_st* stream);

/* Number of SM pairs (two-CTA clusters) gqa_attn_prefill runs on for the
 * current device: the clusters of its kernel that can be resident at once,
 * which the GPC layout can put below half the SM count.  Returns -1 on a CUDA
 * error.  Informational; the library sizes its grid with the same query. */
int gqa_prefill_sm_pairs(void);

/* Human-readable name of a gqa_status value. */
const char* gqa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H */
