// sparse_blocks.cu -- selected-block sparse paged prefill on sm_103a.
//
// Problem ("[Kernel][SM70] Repair #378 on latest main", Changes): each query
// row i (position p = ctx_len - rows + i, 6 query heads sharing 1 KV head,
// D = 256; other groupings run one launch per KV head with up to 16 query
// heads each) attends its own list of selected four-token KV blocks of an fp16
// page-16 cache (block table in physical-page units); the row's own block is
// clamped to p, and an index outside 0 .. p/4 selects nothing.  The page
// converts the blocks into locality-sorted virtual pages for a V100 paged
// kernel; here every row's gather feeds the tensor cores directly:
//
// * Persistent CTAs, one per SM, walk the rows (row = cta, cta + G, ...).  A
//   row's keys come in tiles of 128 (32 blocks); all 6 heads share them.
// * Gather: sixteen warps (eight for K, eight for V; eight in all at head
//   size 128 or for up to 16 heads) issue 16-byte cp.async copies, one
//   warp-wide 512-byte copy per token row, straight into a
//   128B-swizzled smem tile (a warp's copies issue at about 8 bytes per cycle,
//   so the rate grows with the warps that issue them);
//   tokens that are masked (past p, past the list, or a bad id) are
//   zero-filled, so stale cache contents (even NaN) never reach the MMA.
//   Completion is counted on mbarriers (cp.async.mbarrier.arrive.noinc).
// * Swap-AB UMMA with keys as M = 128 and the 6 heads (padded to 16) as N:
//     S^T[128 x 16] = K[128 x 256] . Q^T,  O^T[256 x 16] += V^T . P^T.
// * Softmax across TMEM lanes with a lazily moved per-head reference max
//   (exact cross-lane max only on a row's first tile or when a score exceeds
//   the reference by more than 8 in log2 units; every key thread holds the
//   references in registers); row sums stay per thread until the row ends.
//   The epilogue writes out[i] directly (no split).
//
// * An E4M3 cache (the tail's storage applied to this workload) halves the
//   gathered bytes and has a kernel of its own (sparse_f8_kernel): the codes
//   are gathered unchanged and consumed by FP8 UMMAs (kind::f8f6f4), Q and P
//   entering as three-term E4M3 expansions (see e4m3_umma.cuh); the K scale
//   joins the score scale and the V scale the final 1 / l.
//
// * Short selections: when every row selects at most 16 blocks (64 keys, half
//   a tile), the 6-head kernels take two rows per tile (num_units), their
//   heads side by side in the 16 columns and cross-row scores masked, so the
//   per-row chain of softmax, P.V and epilogue is paid once per two rows.
//
// * Token index warp: block-table lookups (a selected id, then a page id, two
//   dependent loads per key) are taken off the gather warps' path: the index warp
//   resolves each tile's keys to cache token rows ahead of them, through a
//   ring of NI shared-memory slots that the gather warps and the key warps
//   both read (a key whose row is -1 is masked in the copy and the softmax).
// * Selection has set semantics: an id that an earlier position of the row
//   already holds selects nothing more.  The index warp keeps a bitmap of the
//   row's ids seen so far (exact for rows whose own block is below
//   SEEN_BITS; beyond that a hash of the id, with a hit confirmed against the
//   earlier positions), masks the repeat and flags it on the device.
//
// Warp roles: gather warps, then the TMEM owner + UMMA issuer, four key warps
// (softmax + epilogue; thread = TMEM lane) and the token index warp (and, in
// the E4M3 kernel, the warps that build the Q expansions: two, or four for
// two-row units).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <type_traits>

#include "e4m3_umma.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace gqa {
namespace sparse {

constexpr int TILE = 128;            // keys per tile
constexpr int BLK = 4;               // tokens per selected block
constexpr int NP = 16;               // the heads of one launch padded to the UMMA N granule
// Gather warps: a warp-wide 16-byte cp.async copy issues at about 8 bytes per
// cycle per warp, whatever the number of warps (measured: 4 warps move 32, 8
// warps 50, 16 warps 69 bytes per cycle per SM of 512-byte rows from L2), so
// the fp16 kernel gathers with sixteen warps (eight for K, eight for V) at
// head size 256 with 6 heads, eight at head size 128 (sixteen measured no
// faster) and for up to 16 heads (whose key warps need the registers).
template <int HQ, int DH>
constexpr int gather_warps() { return DH == 256 && HQ != NP ? 16 : 8; }
// Warps: gather warps, then the UMMA issuer, four key warps, the index warp.
template <int HQ, int DH>
constexpr int nthreads() { return 32 * (gather_warps<HQ, DH>() + 6); }
constexpr float RESCALE_THRESHOLD = 8.0f;

struct Params {
    const __half* q;
    const __half* kcache;     // fp16 cache
    const __half* vcache;
    const uint8_t* kcache8;   // E4M3 cache
    const uint8_t* vcache8;
    const float* kscale;      // E4M3 scales (device, one fp32 each)
    const float* vscale;
    const int32_t* table;
    const int32_t* sel_idx;
    const int32_t* sel_cnt;
    int max_sel, num_pages, ctx_len, rows, G;
    int log2_page;   // tokens per cache page = 1 << log2_page (8 .. 256)
    int nh;          // query heads of this launch (those of one KV head), <= NP
    int q_stride;    // elements between consecutive rows of q / out (Hq * head size)
    int kv_stride;   // elements between consecutive tokens of the caches (Hkv * head size)
    float scale_log2;
    __half* out;
    unsigned* err;
};

constexpr int PT_BYTES = NP * TILE * 2;                   // 4 KB: 2 chunks [16][64 keys]
constexpr int NI = 8;                                     // token-index ring slots
constexpr int SEEN_BITS = 16384;                          // block ids seen in the row

// smem layout (offsets from a 1024-aligned base) for head size DH (256 or 128)
template <int DH>
struct SL {
    static constexpr int KV_TILE_BYTES = TILE * DH * 2;            // 64 / 32 KB
    static constexpr int OFF_K = 0;                                // 1 K tile
    static constexpr int OFF_V = OFF_K + KV_TILE_BYTES;            // 2 V tiles
    static constexpr int Q_BYTES = NP * DH * 2;                    // DH / 64 chunks [16][64]
    static constexpr int OFF_Q = OFF_V + 2 * KV_TILE_BYTES;        // 2 Q buffers
    static constexpr int OFF_PT = OFF_Q + 2 * Q_BYTES;             // 2 P^T buffers
    static constexpr int OFF_RED = OFF_PT + 2 * PT_BYTES;          // [2][4][NP] tile maxima
    static constexpr int OFF_REDL = OFF_RED + 2 * 4 * NP * 4;      // [2][4][NP] row sums
    static constexpr int OFF_FLAG = OFF_REDL + 2 * 4 * NP * 4;     // [2][4] ints
    static constexpr int OFF_IDX = (OFF_FLAG + 32 + 15) & ~15;     // [NI][TILE] int token rows
    static constexpr int OFF_SEEN = OFF_IDX + NI * TILE * 4;       // [SEEN_BITS / 32] words
    static constexpr int OFF_BAR = (OFF_SEEN + SEEN_BITS / 8 + 7) & ~7;
};
enum {
    B_KFULL = 0,
    B_KEMPTY = 1,
    B_VFULL = 2,   // [2]
    B_VEMPTY = 4,  // [2]
    B_QFULL = 6,   // [2]
    B_QEMPTY = 8,  // [2]
    B_SFULL = 10,  // [2]
    B_PREADY = 12, // [2]
    B_PTEMPTY = 14,// [2]
    B_DRAIN = 16,
    B_GROUP = 17,  // key-thread group barrier
    B_IFULL = 18,       // [NI] token-index slot written
    B_IEMPTY = 18 + NI, // [NI] token-index slot read by the gather and the key warps
    NUM_BARS = 18 + 2 * NI
};
template <int DH>
constexpr int off_tmem() { return SL<DH>::OFF_BAR + NUM_BARS * 8; }
template <int DH>
constexpr int smem_bytes() { return off_tmem<DH>() + 16 + 1024; }
constexpr uint32_t S_COL = 0;        // 2 x NP
constexpr uint32_t O_COL = 2 * NP;   // DH / 128 halves x NP
constexpr uint32_t TMEM_COLS = 128;

__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t u) {
    return r * 128u + ((u ^ (r & 7u)) << 4);
}

// Barrier among the 128 key threads built on an mbarrier (count 128), so that
// it shares the bounded, abort-aware wait of the pipeline barriers: a thread
// that gave up elsewhere cannot leave the others blocked here forever.
__device__ __forceinline__ bool group_sync(uint32_t bar, uint32_t& phase, volatile int* abort,
                                           unsigned* err) {
    mbar_arrive(bar);
    const bool ok = mbar_wait(bar, phase, abort, err);
    phase ^= 1u;
    return ok;
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > 100000000ull) break;
    }
}

// 16-byte async copy global -> shared; src_bytes = 0 zero-fills the destination.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(src_bytes)
                 : "memory");
}

// Arrive on the mbarrier once all of this thread's earlier cp.async copies land.
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ int row_tiles(int cnt) { return (cnt * BLK + TILE - 1) / TILE; }
// Selected blocks of row i, clamped to [0, max_sel]; 0 past the last row.
__device__ __forceinline__ int sel_count(const Params& P, int i) {
    return i < P.rows ? min(max(__ldg(P.sel_cnt + i), 0), P.max_sel) : 0;
}

// Work units.  Without PAIR a unit is one row.  With PAIR (every row selects
// at most 16 blocks, i.e. 64 keys) unit u is rows 2u and 2u + 1 sharing one
// tile: row 2u's keys are keys 0 .. 63 and its heads columns 0 .. 7 of S^T /
// O^T, row 2u + 1's keys 64 .. 127 and columns 8 .. 15; a score of one row's
// head against the other row's key is masked.  Half as many tiles, each
// full, where a row alone would fill half of one.
template <bool PAIR>
__device__ __forceinline__ int num_units(const Params& P) { return PAIR ? (P.rows + 1) / 2 : P.rows; }
template <bool PAIR>
__device__ __forceinline__ int unit_tiles(const Params& P, int u) {
    if (!PAIR) return row_tiles(sel_count(P, u));
    return (sel_count(P, 2 * u) > 0 || sel_count(P, 2 * u + 1) > 0) ? 1 : 0;
}

// ------------------------------------------------------------ token index warp
// (both kernels).  idx: the ring of NI slots of TILE token rows; seen: the
// row's id bitmap; ifull / iempty: the full and empty mbarriers of slot 0
// (each further slot's 8 bytes on).
__device__ __forceinline__ void index_warp(const Params& P, int* idx, uint32_t* seen,
                                           uint32_t ifull, uint32_t iempty,
                                           volatile int* abort_flag) {
    // Same walk as the gather warps (rows of this CTA, tiles of each
    // non-empty row).  Lane l resolves selected position 32 t + l of the
    // row, i.e. keys 4 l .. 4 l + 3 of tile t: id -> set membership ->
    // physical page -> cache token rows, -1 for masked keys (past the
    // list, a bad id, a repeat, or past the row's position).
    const int lane = threadIdx.x & 31;
    const int lp = P.log2_page, pmask = (1 << P.log2_page) - 1;
    uint32_t g = 0;
    bool ok = true;
    for (int i = blockIdx.x; i < P.rows && ok; i += P.G) {
        const int cnt = min(max(__ldg(P.sel_cnt + i), 0), P.max_sel);
        const int nt = row_tiles(cnt);
        if (nt == 0) continue;
        const int p = P.ctx_len - P.rows + i;
        const int own = p / BLK;                     // the row's own block
        const bool exact = own < SEEN_BITS;          // bit = id, no collisions
        const int32_t* sel = P.sel_idx + (size_t)i * P.max_sel;
        for (int w = lane; w < SEEN_BITS / 32; w += 32) seen[w] = 0u;
        __syncwarp();
        for (int t = 0; t < nt; ++t, ++g) {
            const int slot = (int)(g % NI);
            if (!mbar_wait(iempty + 8u * slot, ((g / NI) & 1) ^ 1, abort_flag, P.err)) {
                ok = false;
                break;
            }
            const int li = t * (TILE / BLK) + lane;
            int b = -1;
            bool valid = false;
            if (li < cnt) {
                b = __ldg(sel + li);
                valid = b >= 0 && b <= own;
            }
            const unsigned bad = __ballot_sync(0xffffffffu, li < cnt && !valid);
            if (bad && lane == 0) atomicOr(P.err, kErrBadBlockId);
            // A repeat within this tile: a lower lane holds the same id.
            const unsigned vmask = __ballot_sync(0xffffffffu, valid);
            bool dup = false;
            if (valid) {
                const unsigned same = __match_any_sync(vmask, b);
                dup = (same & ((1u << lane) - 1u)) != 0u;
            }
            // A repeat of an earlier tile: the id's bit is set (exact), or
            // its hash bit is set and an earlier position holds it.
            const uint32_t h = (uint32_t)b & (uint32_t)(SEEN_BITS - 1);
            bool cand = valid && !dup && ((seen[h >> 5] >> (h & 31u)) & 1u);
            if (cand && exact) {
                dup = true;
                cand = false;
            }
            unsigned cm = __ballot_sync(0xffffffffu, cand);
            while (cm) {
                const int src = __ffs(cm) - 1;
                cm &= cm - 1u;
                const int bb = __shfl_sync(0xffffffffu, b, src);
                bool found = false;
                for (int j0 = 0; j0 < t * (TILE / BLK) && !found; j0 += 32)
                    found = __any_sync(0xffffffffu, __ldg(sel + j0 + lane) == bb);
                if (lane == src) dup = found;
            }
            __syncwarp();
            if (valid && !dup) atomicOr(seen + (h >> 5), 1u << (h & 31u));
            if (__ballot_sync(0xffffffffu, dup) && lane == 0) atomicOr(P.err, kErrDupBlockId);
            const bool use = valid && !dup;
            const int tok0 = b * BLK;
            int pg = use ? __ldg(P.table + (tok0 >> lp)) : 0;   // a block never straddles a page
            if (use && (pg < 0 || pg >= P.num_pages)) {
                atomicOr(P.err, kErrBadPageId);
                pg = 0;
            }
            const int r0 = (pg << lp) + (tok0 & pmask);
            int4 r;
            r.x = (use && tok0 + 0 <= p) ? r0 + 0 : -1;
            r.y = (use && tok0 + 1 <= p) ? r0 + 1 : -1;
            r.z = (use && tok0 + 2 <= p) ? r0 + 2 : -1;
            r.w = (use && tok0 + 3 <= p) ? r0 + 3 : -1;
            reinterpret_cast<int4*>(idx + slot * TILE)[lane] = r;
            __syncwarp();   // the set's bits are read by every lane in the next tile
            mbar_arrive(ifull + 8u * slot);
        }
    }
}

// Token-index warp for units of two rows (PAIR; every row selects at most 16
// blocks): lanes 0 .. 15 resolve row 2u's positions 0 .. 15 (keys 0 .. 63 of
// the unit's one tile), lanes 16 .. 31 row 2u + 1's (keys 64 .. 127).  A row's
// whole selection is in this tile, so a repeat is found among the lanes of
// its half alone and no bitmap is needed.
__device__ __forceinline__ void index_warp_pairs(const Params& P, int* idx, uint32_t ifull,
                                                 uint32_t iempty, volatile int* abort_flag) {
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4, li = lane & 15;
    const int lp = P.log2_page, pmask = (1 << P.log2_page) - 1;
    const int nu = (P.rows + 1) / 2;
    uint32_t g = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < nu && ok; u += P.G) {
        const int i = 2 * u + half;            // this half's row (i = rows: none)
        const int cnt = sel_count(P, i);
        if (!__any_sync(0xffffffffu, cnt > 0)) continue;   // the unit has no tile
        const int slot = (int)(g % NI);
        if (!mbar_wait(iempty + 8u * slot, ((g / NI) & 1) ^ 1, abort_flag, P.err)) {
            ok = false;
            break;
        }
        const int p = P.ctx_len - P.rows + i;
        const int own = p / BLK;                   // the row's own block
        int b = -1;
        bool valid = false;
        if (li < cnt) {
            b = __ldg(P.sel_idx + (size_t)i * P.max_sel + li);
            valid = b >= 0 && b <= own;
        }
        const unsigned bad = __ballot_sync(0xffffffffu, li < cnt && !valid);
        if (bad && lane == 0) atomicOr(P.err, kErrBadBlockId);
        // A repeat: a lower lane of the same row holds the same id.
        const unsigned vmask = __ballot_sync(0xffffffffu, valid);
        bool dup = false;
        if (valid) {
            const unsigned same = __match_any_sync(vmask, (b << 1) | half);
            dup = (same & ((1u << lane) - 1u)) != 0u;
        }
        if (__ballot_sync(0xffffffffu, dup) && lane == 0) atomicOr(P.err, kErrDupBlockId);
        const bool use = valid && !dup;
        const int tok0 = b * BLK;
        int pg = use ? __ldg(P.table + (tok0 >> lp)) : 0;   // a block never straddles a page
        if (use && (pg < 0 || pg >= P.num_pages)) {
            atomicOr(P.err, kErrBadPageId);
            pg = 0;
        }
        const int r0 = (pg << lp) + (tok0 & pmask);
        int4 r;
        r.x = (use && tok0 + 0 <= p) ? r0 + 0 : -1;
        r.y = (use && tok0 + 1 <= p) ? r0 + 1 : -1;
        r.z = (use && tok0 + 2 <= p) ? r0 + 2 : -1;
        r.w = (use && tok0 + 3 <= p) ? r0 + 3 : -1;
        reinterpret_cast<int4*>(idx + slot * TILE)[lane] = r;
        __syncwarp();
        mbar_arrive(ifull + 8u * slot);
        ++g;
    }
}

// fp16 cache.  HQ: heads per launch known at compile time (6), or NP with the
// count read from P.nh (any grouping up to 16 query heads per KV head).  DH:
// head size, 256 or 128.  PAIR: units of two rows per tile (see num_units).
template <int HQ, int DH, bool PAIR>
__global__ void __launch_bounds__(nthreads<HQ, DH>(), 1) sparse_kernel(const Params P) {
    static_assert(!PAIR || HQ <= 8, "two rows' heads in 16 columns");
    using L = SL<DH>;
    const int NU = num_units<PAIR>(P);
    constexpr int HALVES = DH / 128;   // 128-d halves of a row (one M = 128 P.V each)
    constexpr int KV_TILE_BYTES = L::KV_TILE_BYTES;
    constexpr int OFF_K = L::OFF_K, OFF_V = L::OFF_V, Q_BYTES = L::Q_BYTES, OFF_Q = L::OFF_Q;
    constexpr int OFF_PT = L::OFF_PT, OFF_RED = L::OFF_RED, OFF_REDL = L::OFF_REDL;
    constexpr int OFF_FLAG = L::OFF_FLAG, OFF_IDX = L::OFF_IDX;
    constexpr int OFF_SEEN = L::OFF_SEEN, OFF_BAR = L::OFF_BAR, OFF_TMEM = off_tmem<DH>();
    const int nh = (HQ == NP) ? P.nh : HQ;
    const size_t q_stride = (HQ == NP) ? (size_t)P.q_stride : (size_t)HQ * DH;
    // Tile buffers (fp16, whatever the cache holds): one K tile and two V
    // tiles (the K tile is free again as soon as its Q.K^T is done, a V tile
    // only after the softmax and P.V).
    constexpr int NVB = 2;
    constexpr uint32_t KOFF = OFF_K;
    constexpr uint32_t VOFF = OFF_V;
    constexpr int NGW = gather_warps<HQ, DH>();
    constexpr int NTHREADS = nthreads<HQ, DH>();
    constexpr int MMA_WARP = NGW, KEY_WARP0 = NGW + 1, IDX_WARP = NGW + 5;
    // Arrivals per K or V tile: every thread of the operand's NGW / 2 gather warps.
    constexpr int NGATHER = 32 * (NGW / 2);
    constexpr int NQLOAD = 128;   // threads that load Q and arrive on its barrier
    constexpr uint32_t IDESC_QK = idesc_f16_f32(128, NP, false, false);
    constexpr uint32_t IDESC_PV = idesc_f16_f32(128, NP, true, false);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (sbase - smem_u32(smem_raw));
    float* red = reinterpret_cast<float*>(gbase + OFF_RED);
    float* redl = reinterpret_cast<float*>(gbase + OFF_REDL);
    volatile int* flags = reinterpret_cast<volatile int*>(gbase + OFF_FLAG);
    const uint32_t bars = sbase + OFF_BAR;
    uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(gbase + OFF_TMEM);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_ptr + 1);
    auto bar = [&](int i) { return bars + 8u * i; };
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar(B_KFULL), NGATHER);
        mbar_init(bar(B_KEMPTY), 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_VFULL + b), NGATHER);
            mbar_init(bar(B_VEMPTY + b), 1);
            mbar_init(bar(B_QFULL + b), NQLOAD);
            mbar_init(bar(B_QEMPTY + b), 1);
            mbar_init(bar(B_SFULL + b), 1);
            mbar_init(bar(B_PREADY + b), 128);
            mbar_init(bar(B_PTEMPTY + b), 1);
        }
        mbar_init(bar(B_DRAIN), 1);
        mbar_init(bar(B_GROUP), 128);
        for (int b = 0; b < NI; ++b) {
            mbar_init(bar(B_IFULL + b), 32);
            mbar_init(bar(B_IEMPTY + b), 32 * NGW + 128);   // gather and key threads
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    // Zero both Q buffers once (rows 6..15 stay zero).
    for (int u = threadIdx.x; u < 2 * Q_BYTES / 16; u += NTHREADS)
        *reinterpret_cast<uint4*>(gbase + OFF_Q + u * 16) = make_uint4(0, 0, 0, 0);
    if (warp == MMA_WARP) {
        tmem_alloc(smem_u32(tmem_ptr), TMEM_COLS);
        tmem_relinquish();
    }
    fence_async_shared();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_ptr;

    if (warp < NGW) {
        // ------------------------------------------------------------ gather
        const int gt = threadIdx.x;        // 0 .. 32 NGW - 1
        const int* idx = reinterpret_cast<const int*>(gbase + OFF_IDX);
        const size_t tok_stride = HQ == NP ? (size_t)P.kv_stride : (size_t)DH;
        // Cache row offset of key kbase + lane of tile-counter position gg, read
        // from the index ring; tok < 0 for a masked key.
        auto take_index = [&](uint32_t gg, int kbase, int& tok, size_t& row) -> bool {
            const int slot = (int)(gg % NI);
            if (!mbar_wait(bar(B_IFULL + slot), (gg / NI) & 1, abort_flag, P.err)) return false;
            tok = idx[slot * TILE + min(kbase + lane, TILE - 1)];
            mbar_arrive(bar(B_IEMPTY + slot));
            row = tok >= 0 ? (size_t)tok * tok_stride : 0;
            return true;
        };
        uint32_t g = 0;                     // global tile counter
        int rloc = 0;                       // non-empty rows handled so far
        bool ok = true;
        for (int un = blockIdx.x; un < NU && ok; un += P.G) {
            const int nt = unit_tiles<PAIR>(P, un);
            const int i = un;   // the row (without PAIR)
            if (nt == 0) continue;
            // Q row i (nh heads x DH d) -> Q buffer rloc & 1, rows 0 .. nh - 1
            // (with PAIR rows 2un and 2un + 1, head h of row r at Q row
            // 8 r + h), by the NQLOAD threads that count on QFULL (the first
            // gather warps).
            const int qb = rloc & 1;
            if (gt < NQLOAD) {
                if (!mbar_wait(bar(B_QEMPTY + qb), ((rloc >> 1) & 1) ^ 1, abort_flag, P.err)) {
                    ok = false;
                    break;
                }
                const int ne = PAIR ? 2 * HQ : nh;   // head rows to load
                for (int v = gt; v < ne * (DH / 8); v += NQLOAD) {
                    const int e = v / (DH / 8), c16 = v % (DH / 8);
                    const int sr = PAIR ? e / HQ : 0, h = e - sr * HQ;
                    const int row = PAIR ? 2 * un + sr : i;
                    if (row >= P.rows) continue;   // the missing second row of the last unit
                    const uint32_t dst = sbase + OFF_Q + qb * Q_BYTES + (c16 / 8) * (NP * 128) +
                                         sw128(sr * 8 + h, c16 % 8);
                    cp_async16(dst, P.q + (size_t)row * q_stride + h * DH + c16 * 8, 16);
                }
                cp_async_arrive(bar(B_QFULL + qb));
            }
            ++rloc;
            // Warps 0 .. NGW / 2 - 1 gather K and the others V, each warp KPW
            // keys of every tile, so the K stream runs ahead of the V stream
            // (K's single buffer frees once its Q.K^T is done, V's two buffers
            // after each P.V).
            constexpr int KW = NGW / 2;        // warps per operand
            constexpr int KPW = TILE / KW;     // keys per warp: 32 or 16
            static_assert(KPW <= 32 && TILE == KPW * KW, "keys per warp");
            const bool kg = warp < KW;
            const int kbase = (warp % KW) * KPW;
            // fp16: a key's row is DH * 2 bytes, one warp-wide 16-byte-per-lane
            // copy per 512 / (DH * 2) keys, straight into the swizzled tile.
            constexpr int LPK = DH / 8;       // lanes per key row: 32 or 16
            constexpr int KPI = 32 / LPK;     // keys per copy instruction: 1 or 2
            const int ul = lane % LPK;        // lane covers d = 8 ul .. 8 ul + 7
            const __half* cache = kg ? P.kcache : P.vcache;
            for (int t = 0; t < nt && ok; ++t, ++g) {
                int tok1;
                size_t row1;
                if (!take_index(g, kbase, tok1, row1)) {
                    ok = false;
                    break;
                }
                // (lanes KPW .. 31 read keys of the next warp; their values are unused)
                uint32_t tile, fullb;
                if (kg) {
                    if (!mbar_wait(bar(B_KEMPTY), (g & 1) ^ 1, abort_flag, P.err)) {
                        ok = false;
                        break;
                    }
                    tile = sbase + OFF_K;
                    fullb = bar(B_KFULL);
                } else {
                    const int vb = g & 1;
                    if (!mbar_wait(bar(B_VEMPTY + vb), ((g >> 1) & 1) ^ 1, abort_flag, P.err)) {
                        ok = false;
                        break;
                    }
                    tile = sbase + OFF_V + vb * KV_TILE_BYTES;
                    fullb = bar(B_VFULL + vb);
                }
#pragma unroll 4
                for (int e = 0; e < KPW / KPI; ++e) {
                    const int src = KPI * e + lane / LPK;   // lane holding this key's row
                    const int key = kbase + src;
                    const int tok = __shfl_sync(0xffffffffu, tok1, src);
                    const size_t row = __shfl_sync(0xffffffffu, row1, src);
                    // chunk ul / 8, unit ul % 8 of the key's swizzled row
                    const uint32_t dst = tile + (ul >> 3) * (TILE * 128) + sw128(key, ul & 7);
                    const __half* sp = tok >= 0 ? cache + row + ul * 8 : cache;
                    cp_async16(dst, sp, tok >= 0 ? 16u : 0u);
                }
                cp_async_arrive(fullb);
            }
        }
        if (!ok) asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------------------ UMMA issuer
        if (lane == 0) {
            uint32_t g = 0;
            int rloc = 0;
            bool ok = true;
            auto issue_pv = [&](uint32_t x, bool first) -> bool {
                if (!mbar_wait(bar(B_PREADY + (x & 1)), (x >> 1) & 1, abort_flag, P.err))
                    return false;
                const int vb = (int)(x % NVB);
                if (!mbar_wait(bar(B_VFULL + vb), (x / NVB) & 1, abort_flag, P.err)) return false;
                fence_async_shared();
                tc_fence_after();
                const uint32_t pt = sbase + OFF_PT + (x & 1) * PT_BYTES;
#pragma unroll
                for (int h = 0; h < HALVES; ++h) {
#pragma unroll
                    for (int ks = 0; ks < TILE / 16; ++ks) {
                        const uint64_t a = sdesc_sw128(sbase + VOFF + vb * KV_TILE_BYTES +
                                                           (2 * h) * (TILE * 128) +
                                                           ks * 2048,
                                                       TILE * 128, 1024);
                        const uint64_t b =
                            sdesc_sw128(pt + (ks / 4) * (NP * 128) + (ks % 4) * 32, 16, 1024);
                        umma_ss(tmem + O_COL + h * NP, a, b, IDESC_PV, (!first || ks > 0));
                    }
                }
                umma_commit(bar(B_PTEMPTY + (x & 1)));
                umma_commit(bar(B_VEMPTY + vb));
                return true;
            };
            for (int un = blockIdx.x; un < NU && ok; un += P.G) {
                const int nt = unit_tiles<PAIR>(P, un);
                if (nt == 0) continue;
                const int qb = rloc & 1;
                if (!mbar_wait(bar(B_QFULL + qb), (rloc >> 1) & 1, abort_flag, P.err)) {
                    ok = false;
                    break;
                }
                ++rloc;
                // cp.async writes are generic-proxy writes; order them before UMMA reads.
                fence_async_shared();
                const uint32_t g0 = g;
                for (int t = 0; t < nt; ++t, ++g) {
                    if (!mbar_wait(bar(B_KFULL), g & 1, abort_flag, P.err)) {
                        ok = false;
                        break;
                    }
                    fence_async_shared();
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < DH / 16; ++kk) {
                        const uint64_t a = sdesc_sw128(sbase + KOFF +
                                                           (kk / 4) * (TILE * 128) + (kk % 4) * 32,
                                                       16, 1024);
                        const uint64_t b = sdesc_sw128(sbase + OFF_Q + qb * Q_BYTES +
                                                           (kk / 4) * (NP * 128) + (kk % 4) * 32,
                                                       16, 1024);
                        umma_ss(tmem + S_COL + (g & 1) * NP, a, b, IDESC_QK, kk > 0);
                    }
                    umma_commit(bar(B_SFULL + (g & 1)));
                    umma_commit(bar(B_KEMPTY));
                    if (t == nt - 1) umma_commit(bar(B_QEMPTY + qb));
                    if (t >= 1 && !(ok = issue_pv(g - 1, g - 1 == g0))) break;
                }
                if (ok) ok = issue_pv(g - 1, g - 1 == g0);
            }
            if (!ok) {
                umma_commit(bar(B_DRAIN));
                drain_wait(bar(B_DRAIN), 0);
            }
        }
    } else if (warp < KEY_WARP0 + 4) {
        // ------------------------------------------------------------ key warps
        // Each thread keeps every head's reference max in registers: after a
        // vote fires, the warps' partial maxima go through shared memory and
        // one barrier, and every thread derives the same new references.
        const int wq = warp & 3;
        const int k = wq * 32 + lane;
        const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
        const float sl2 = P.scale_log2;
        uint32_t g = 0;
        uint32_t gphase = 0;
        int rpar = 0;   // parity of the non-empty rows handled (row-sum slot)
        bool ok = true;
        if constexpr (PAIR) {
            // Units of two rows, one tile each: S^T column c is head c & 7 of
            // row 2un + (c >> 3); key k belongs to row 2un + (k >> 6).
            for (int un = blockIdx.x; un < NU && ok; un += P.G) {
                const int i0 = 2 * un;
                if (unit_tiles<PAIR>(P, un) == 0) {
                    // Nothing selected in either row: both outputs are zero.
                    for (int sr = 0; sr < 2 && i0 + sr < P.rows; ++sr)
                        for (int v = k; v < HQ * (DH / 8); v += 128)
                            reinterpret_cast<uint4*>(P.out + (size_t)(i0 + sr) * q_stride)[v] =
                                make_uint4(0, 0, 0, 0);
                    continue;
                }
                const int b = g & 1;
                bool masked;
                {
                    // The index warp's verdict on this key (-1: masked).
                    const int slot = (int)(g % NI);
                    ok = mbar_wait(bar(B_IFULL + slot), (g / NI) & 1, abort_flag, P.err);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    masked = reinterpret_cast<const int*>(gbase + OFF_IDX)[slot * TILE + k] < 0;
                    mbar_arrive(bar(B_IEMPTY + slot));
                }
                ok = mbar_wait(bar(B_SFULL + b), (g >> 1) & 1, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                const int kr = k >> 6;   // the unit's row this key belongs to
                float s[NP];
                {
                    uint32_t r[NP];
                    tmem_ld16(t_lane + S_COL + b * NP, r);
                    tmem_ld_wait<NP>(r);
#pragma unroll
                    for (int c = 0; c < NP; ++c)
                        s[c] = (masked || (c >> 3) != kr || (c & 7) >= HQ) ? -INFINITY
                                                                           : __uint_as_float(r[c]) * sl2;
                }
                // The unit's one tile: each column's exact max is its reference.
                float* rd = red + (g & 1) * (4 * NP);
#pragma unroll
                for (int c = 0; c < NP; ++c) {
                    if ((c & 7) >= HQ) continue;
                    float m = s[c];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                    if (lane == 0) rd[wq * NP + c] = m;
                }
                ok = group_sync(bar(B_GROUP), gphase, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                // P^T buffer b is free once the P.V two tiles back has completed.
                ok = mbar_wait(bar(B_PTEMPTY + b), ((g >> 1) & 1) ^ 1, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                float pl[NP];
                {
                    uint8_t* pt = gbase + OFF_PT + b * PT_BYTES;
                    const int kc = k >> 6, kin = k & 63;
#pragma unroll
                    for (int c = 0; c < NP; ++c) {
                        pl[c] = 0.f;
                        if ((c & 7) < HQ) {
                            const float tmax = fmaxf(fmaxf(rd[c], rd[NP + c]),
                                                     fmaxf(rd[2 * NP + c], rd[3 * NP + c]));
                            pl[c] = ex2(s[c] - (tmax == -INFINITY ? 0.f : tmax));
                        }
                        const uint32_t off = kc * (NP * 128) + sw128(c, kin >> 3) + (kin & 7) * 2;
                        *reinterpret_cast<__half*>(pt + off) = __float2half_rn(pl[c]);
                    }
                }
                fence_async_shared();
                mbar_arrive(bar(B_PREADY + b));
                // Row sums per column (this tile is the unit's only one), while
                // the P.V runs: warp sums -> redl (slot of this unit's parity).
                float* rl = redl + rpar * (4 * NP);
                rpar ^= 1;
#pragma unroll
                for (int c = 0; c < NP; ++c) {
                    if ((c & 7) >= HQ) continue;
                    float v = pl[c];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == 0) rl[wq * NP + c] = v;
                }
                // ---------------------------------------------------------- unit epilogue
                const uint32_t x = g++;
                ok = mbar_wait(bar(B_PTEMPTY + (x & 1)), (x >> 1) & 1, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                ok = group_sync(bar(B_GROUP), gphase, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                float inv[NP];
#pragma unroll
                for (int c = 0; c < NP; ++c) {
                    const float l = (rl[c] + rl[NP + c]) + (rl[2 * NP + c] + rl[3 * NP + c]);
                    inv[c] = ((c & 7) < HQ && l > 0.f) ? 1.0f / l : 0.f;
                }
#pragma unroll
                for (int h = 0; h < HALVES; ++h) {
                    uint32_t r[NP];
                    tmem_ld16(t_lane + O_COL + h * NP, r);
                    tmem_ld_wait<NP>(r);
                    const int d = h * 128 + k;
#pragma unroll
                    for (int c = 0; c < NP; ++c) {
                        const int row = i0 + (c >> 3);
                        if ((c & 7) < HQ && row < P.rows)
                            P.out[(size_t)row * q_stride + (c & 7) * DH + d] =
                                __float2half_rn(__uint_as_float(r[c]) * inv[c]);
                    }
                }
            }
        } else {
            for (int un = blockIdx.x; un < NU && ok; un += P.G) {
                const int nt = unit_tiles<PAIR>(P, un);
                const int i = un;   // the row (without PAIR)
                if (nt == 0) {
                    // Nothing selected: the row's output is zero.
                    for (int u = k; u < nh * (DH / 8); u += 128)
                        reinterpret_cast<uint4*>(P.out + (size_t)i * q_stride)[u] = make_uint4(0, 0, 0, 0);
                    continue;
                }
                float mr[HQ], lpart[HQ];
    #pragma unroll
                for (int c = 0; c < HQ; ++c) {
                    mr[c] = -INFINITY;
                    lpart[c] = 0.f;
                }
                for (int t = 0; t < nt; ++t, ++g) {
                    const int b = g & 1;
                    bool masked;
                    {
                        // The index warp's verdict on this key (-1: masked).
                        const int slot = (int)(g % NI);
                        ok = mbar_wait(bar(B_IFULL + slot), (g / NI) & 1, abort_flag, P.err);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                        masked = reinterpret_cast<const int*>(gbase + OFF_IDX)[slot * TILE + k] < 0;
                        mbar_arrive(bar(B_IEMPTY + slot));
                    }
                    ok = mbar_wait(bar(B_SFULL + b), (g >> 1) & 1, abort_flag, P.err);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after();
                    float s[NP];
                    {
                        uint32_t r[NP];
                        tmem_ld16(t_lane + S_COL + b * NP, r);
                        tmem_ld_wait<NP>(r);
    #pragma unroll
                        for (int c = 0; c < NP; ++c) s[c] = masked ? -INFINITY : __uint_as_float(r[c]) * sl2;
                    }
                    // A row's first tile always takes the exact max (its references
                    // are -inf); later tiles only when a score crosses its reference.
                    bool any = t == 0;
                    if (!any) {
                        bool exceed = false;
    #pragma unroll
                        for (int c = 0; c < HQ; ++c)
                            if (c < nh) exceed |= s[c] > mr[c] + RESCALE_THRESHOLD;
                        const unsigned vote = __ballot_sync(0xffffffffu, exceed);
                        volatile int* fl = flags + (g & 1) * 4;
                        if (lane == 0) fl[wq] = vote != 0;
                        ok = group_sync(bar(B_GROUP), gphase, abort_flag, P.err);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                        any = fl[0] | fl[1] | fl[2] | fl[3];
                    }
                    if (any) {
                        // The tile's max per head: warp maxima -> red (its slot of
                        // this tile parity) -> one barrier -> every thread.
                        float* rd = red + (g & 1) * (4 * NP);
    #pragma unroll
                        for (int c = 0; c < HQ; ++c) {
                            if (c >= nh) break;
                            float m = s[c];
    #pragma unroll
                            for (int o = 16; o > 0; o >>= 1)
                                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                            if (lane == 0) rd[wq * NP + c] = m;
                        }
                        ok = group_sync(bar(B_GROUP), gphase, abort_flag, P.err);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                        float f[HQ];
    #pragma unroll
                        for (int c = 0; c < HQ; ++c) {
                            f[c] = 1.0f;
                            if (c < nh) {
                                const float tmax = fmaxf(fmaxf(rd[c], rd[NP + c]),
                                                         fmaxf(rd[2 * NP + c], rd[3 * NP + c]));
                                if (tmax > mr[c] + RESCALE_THRESHOLD) {
                                    f[c] = (mr[c] == -INFINITY) ? 0.f : ex2(mr[c] - tmax);
                                    mr[c] = tmax;
                                }
                            }
                        }
                        if (t > 0) {
                            // O^T must hold every earlier P.V of the row before it is rescaled.
                            const uint32_t x = g - 1;
                            ok = mbar_wait(bar(B_PTEMPTY + (x & 1)), (x >> 1) & 1, abort_flag, P.err);
                            ok = __all_sync(0xffffffffu, ok);
                            if (!ok) break;
                            tc_fence_after();
    #pragma unroll
                            for (int h = 0; h < HALVES; ++h) {
                                uint32_t r[NP];
                                tmem_ld16(t_lane + O_COL + h * NP, r);
                                tmem_ld_wait<NP>(r);
    #pragma unroll
                                for (int c = 0; c < HQ; ++c)
                                    r[c] = __float_as_uint(__uint_as_float(r[c]) * f[c]);
                                tmem_st16(t_lane + O_COL + h * NP, r);
                            }
                            tmem_st_wait();
                        }
    #pragma unroll
                        for (int c = 0; c < HQ; ++c) lpart[c] *= f[c];
                    }
                    ok = mbar_wait(bar(B_PTEMPTY + b), ((g >> 1) & 1) ^ 1, abort_flag, P.err);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    uint8_t* pt = gbase + OFF_PT + b * PT_BYTES;
                    const int kc = k >> 6, kin = k & 63;
    #pragma unroll
                    for (int c = 0; c < NP; ++c) {
                        float p = 0.f;
                        if (c < HQ && c < nh) {
                            const float m = mr[c < HQ ? c : 0];
                            p = ex2(s[c] - (m == -INFINITY ? 0.f : m));
                            lpart[c < HQ ? c : 0] += p;
                        }
                        const uint32_t off = kc * (NP * 128) + sw128(c, kin >> 3) + (kin & 7) * 2;
                        *reinterpret_cast<__half*>(pt + off) = __float2half_rn(p);
                    }
                    fence_async_shared();
                    mbar_arrive(bar(B_PREADY + b));
                }
                if (!ok) break;
                // ---------------------------------------------------------- row epilogue
                const uint32_t x = g - 1;
                ok = mbar_wait(bar(B_PTEMPTY + (x & 1)), (x >> 1) & 1, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                // Row sums: warp sums -> redl (its slot of this row parity) -> one
                // barrier.  The next write to the same slot comes two rows later,
                // behind barriers every thread passes after its reads here.
                float* rl = redl + rpar * (4 * NP);
                rpar ^= 1;
    #pragma unroll
                for (int c = 0; c < HQ; ++c) {
                    if (c >= nh) break;
                    float v = lpart[c];
    #pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == 0) rl[wq * NP + c] = v;
                }
                ok = group_sync(bar(B_GROUP), gphase, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                float inv[HQ];
    #pragma unroll
                for (int c = 0; c < HQ; ++c) {
                    const float l = (rl[c] + rl[NP + c]) + (rl[2 * NP + c] + rl[3 * NP + c]);
                    inv[c] = l > 0.f ? 1.0f / l : 0.f;
                }
    #pragma unroll
                for (int h = 0; h < HALVES; ++h) {
                    uint32_t r[NP];
                    tmem_ld16(t_lane + O_COL + h * NP, r);
                    tmem_ld_wait<NP>(r);
                    const int d = h * 128 + k;
    #pragma unroll
                    for (int c = 0; c < HQ; ++c)
                        if (c < nh)
                            P.out[(size_t)i * q_stride + c * DH + d] =
                                __float2half_rn(__uint_as_float(r[c]) * inv[c]);
                }
            }
        }
    }

    if (warp == IDX_WARP) {
        if constexpr (PAIR)
            index_warp_pairs(P, reinterpret_cast<int*>(gbase + OFF_IDX), bar(B_IFULL),
                             bar(B_IEMPTY), abort_flag);
        else
            index_warp(P, reinterpret_cast<int*>(gbase + OFF_IDX),
                       reinterpret_cast<uint32_t*>(gbase + OFF_SEEN), bar(B_IFULL), bar(B_IEMPTY),
                       abort_flag);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ======================================================================
// E4M3 cache: raw codes on the FP8 tensor cores.
//
// The gather copies a selected token's E4M3 code row (DH bytes) unchanged
// into a 128B-swizzled tile, in 128-byte halves of d, the layout a TMA copy
// of a cache page would give.  Q.K^T and P.V then run as tcgen05.mma
// kind::f8f6f4 on those bytes, so nothing is decoded: Q (one scale per head,
// x / qs within +-256) and P (<= 256) enter as three-term E4M3 expansions laid
// side by side along N (term e of head c is row e * TS + c of the operand),
// and the key threads combine the three partial products of S^T and O^T.
// The K scale joins the score scale and the V scale the final 1 / l.
// A moved reference max sits REF_SHIFT below the tile's max, so that P stays
// far above the expansion's floor of 2^-19 (the paged tail's rule).
// Warps: gather warps (half K, half V), the UMMA issuer, four key warps, the
// token index warp, then the warps that build each unit's Q expansion one
// unit ahead (two Q buffers).  Two K and two V buffers: the gather of
// tile t + 1 never waits for the Q.K^T of tile t.
// ======================================================================
// Warps that build the Q expansions: two for a row's heads, four for a
// unit of two rows (twelve head rows per unit).
template <bool PAIR>
constexpr int f8_qwarps() { return PAIR ? 4 : 2; }
constexpr int F8_NKB = 2, F8_NVB = 2;   // K / V tile buffers
constexpr int F8_NQB = 2;               // Q expansion buffers
// Rows per expansion term (the heads of the launch, padded to 8; with PAIR
// the heads of two rows, 8 columns each) and the UMMA N: three terms, rounded
// up to the N granule of 16.
template <int HQ, bool PAIR>
constexpr int f8_ts() { return (HQ == NP || PAIR) ? NP : 8; }
template <int HQ, bool PAIR>
constexpr int f8_n() { return (3 * f8_ts<HQ, PAIR>() + 15) / 16 * 16; }
// Half the bytes of the fp16 rows: eight gather warps move a tile's codes in
// about the time sixteen take for fp16.
template <int HQ, int DH>
constexpr int f8_gather_warps() { return 8; }
template <int HQ, int DH, bool PAIR>
constexpr int f8_nthreads() { return 32 * (f8_gather_warps<HQ, DH>() + 6 + f8_qwarps<PAIR>()); }
enum {
    F_KFULL = 0,      // [F8_NKB]
    F_KEMPTY = 2,     // [F8_NKB]
    F_VFULL = 4,      // [F8_NVB]
    F_VEMPTY = 7,     // [F8_NVB]
    F_QFULL = 10,     // [F8_NQB]
    F_QEMPTY = 13,    // [F8_NQB] the row's last Q.K^T and its key threads' epilogue
    F_SFULL = 16,     // [2]
    F_PREADY = 18,    // [2]
    F_PTEMPTY = 20,   // [2]
    F_DRAIN = 22,
    F_GROUP = 23,
    F_IFULL = 24,          // [NI]
    F_IEMPTY = 24 + NI,    // [NI]
    F_NUM_BARS = 24 + 2 * NI
};
static_assert(F8_NKB <= 2 && F8_NVB <= 3 && F8_NQB <= 3, "barrier slots");
// smem layout (offsets from a 1024-aligned base)
template <int HQ, int DH, bool PAIR>
struct SL8 {
    static constexpr int TS = f8_ts<HQ, PAIR>();
    static constexpr int N3 = f8_n<HQ, PAIR>();
    static constexpr int RAW_TILE = TILE * DH;                     // 32 / 16 KB of codes
    static constexpr int OFF_K = 0;                                // [F8_NKB][DH / 128][TILE][128]
    static constexpr int OFF_V = OFF_K + F8_NKB * RAW_TILE;        // [F8_NVB][DH / 128][TILE][128]
    static constexpr int Q_BYTES = N3 * DH;                        // [DH / 128][N3][128]
    static constexpr int OFF_Q = OFF_V + F8_NVB * RAW_TILE;        // F8_NQB Q expansions
    static constexpr int PT_BYTES = N3 * TILE;                     // [N3][128 keys]
    static constexpr int OFF_PT = OFF_Q + F8_NQB * Q_BYTES;        // 2 P^T expansions
    static constexpr int OFF_QS = OFF_PT + 2 * PT_BYTES;           // [F8_NQB][NP] Q scales
    static constexpr int OFF_RED = OFF_QS + F8_NQB * NP * 4;       // [2][4][NP] tile maxima
    static constexpr int OFF_REDL = OFF_RED + 2 * 4 * NP * 4;      // [2][4][NP] row sums
    static constexpr int OFF_FLAG = OFF_REDL + 2 * 4 * NP * 4;     // [2][4] ints
    static constexpr int OFF_IDX = (OFF_FLAG + 32 + 15) & ~15;     // [NI][TILE] token rows
    static constexpr int OFF_SEEN = OFF_IDX + NI * TILE * 4;
    static constexpr int OFF_BAR = (OFF_SEEN + SEEN_BITS / 8 + 7) & ~7;
    static constexpr int OFF_TMEM = OFF_BAR + F_NUM_BARS * 8;
    static constexpr int SMEM = OFF_TMEM + 16 + 1024;
    static constexpr uint32_t S_COL = 0;            // 2 x N3
    static constexpr uint32_t O_COL = 2 * N3;       // DH / 128 halves x N3
    static_assert(OFF_Q % 1024 == 0 && OFF_PT % 1024 == 0 && Q_BYTES % 1024 == 0 &&
                  PT_BYTES % 1024 == 0, "swizzle atoms");
    static_assert(O_COL + (DH / 128) * N3 <= 256, "tensor memory columns");
};
constexpr uint32_t F8_TMEM_COLS = 256;

template <int HQ, int DH, bool PAIR>
__global__ void __launch_bounds__(f8_nthreads<HQ, DH, PAIR>(), 1) sparse_f8_kernel(const Params P) {
    static_assert(!PAIR || HQ <= 8, "two rows' heads in 16 columns");
    using L = SL8<HQ, DH, PAIR>;
    const int NU = num_units<PAIR>(P);
    constexpr int HALVES = DH / 128;
    constexpr int TS = L::TS, N3 = L::N3, RAW_TILE = L::RAW_TILE;
    constexpr int NGW = f8_gather_warps<HQ, DH>();
    constexpr int NTHREADS = f8_nthreads<HQ, DH, PAIR>();
    constexpr int F8_QWARPS = f8_qwarps<PAIR>();
    constexpr int MMA_WARP = NGW, KEY_WARP0 = NGW + 1, IDX_WARP = NGW + 5, Q_WARP0 = NGW + 6;
    constexpr int NGATHER = 32 * (NGW / 2);   // arrivals per K or V tile
    // E4M3 x E4M3 -> f32 (format fields 0 = E4M3 for kind::f8f6f4); A = K
    // (K-major) for Q.K^T, A = V^T (MN-major) for P.V.
    constexpr uint32_t IDESC_QK = idesc_f16_f32(128, N3, false, false);
    constexpr uint32_t IDESC_PV = idesc_f16_f32(128, N3, true, false);
    const int nh = (HQ == NP) ? P.nh : HQ;
    const size_t q_stride = (HQ == NP) ? (size_t)P.q_stride : (size_t)HQ * DH;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (sbase - smem_u32(smem_raw));
    float* qs = reinterpret_cast<float*>(gbase + L::OFF_QS);
    float* red = reinterpret_cast<float*>(gbase + L::OFF_RED);
    float* redl = reinterpret_cast<float*>(gbase + L::OFF_REDL);
    volatile int* flags = reinterpret_cast<volatile int*>(gbase + L::OFF_FLAG);
    const uint32_t bars = sbase + L::OFF_BAR;
    uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(gbase + L::OFF_TMEM);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_ptr + 1);
    auto bar = [&](int i) { return bars + 8u * i; };
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int b = 0; b < F8_NKB; ++b) {
            mbar_init(bar(F_KFULL + b), NGATHER);
            mbar_init(bar(F_KEMPTY + b), 1);
        }
        for (int b = 0; b < F8_NVB; ++b) {
            mbar_init(bar(F_VFULL + b), NGATHER);
            mbar_init(bar(F_VEMPTY + b), 1);
        }
        for (int b = 0; b < F8_NQB; ++b) {
            mbar_init(bar(F_QFULL + b), 32 * F8_QWARPS);
            mbar_init(bar(F_QEMPTY + b), 2);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(F_SFULL + b), 1);
            mbar_init(bar(F_PREADY + b), 128);
            mbar_init(bar(F_PTEMPTY + b), 1);
        }
        mbar_init(bar(F_DRAIN), 1);
        mbar_init(bar(F_GROUP), 128);
        for (int b = 0; b < NI; ++b) {
            mbar_init(bar(F_IFULL + b), 32);
            mbar_init(bar(F_IEMPTY + b), 32 * NGW + 128);   // gather and key threads
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    // Zero the Q and P^T expansions once: rows no head writes (heads past nh,
    // the padding of N) stay zero.
    for (int u = threadIdx.x; u < (F8_NQB * L::Q_BYTES + 2 * L::PT_BYTES) / 16; u += NTHREADS)
        *reinterpret_cast<uint4*>(gbase + L::OFF_Q + u * 16) = make_uint4(0, 0, 0, 0);
    if (warp == MMA_WARP) {
        tmem_alloc(smem_u32(tmem_ptr), F8_TMEM_COLS);
        tmem_relinquish();
    }
    fence_async_shared();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_ptr;

    if (warp < NGW) {
        // ------------------------------------------------------------ gather
        // Warps 0 .. NGW / 2 - 1 copy K code rows, the others V, KPW keys of
        // every tile each; a code row is DH bytes, LPK lanes of 16 bytes.
        const int* idx = reinterpret_cast<const int*>(gbase + L::OFF_IDX);
        const size_t tok_stride = HQ == NP ? (size_t)P.kv_stride : (size_t)DH;
        constexpr int KW = NGW / 2;
        constexpr int KPW = TILE / KW;
        static_assert(KPW <= 32 && TILE == KPW * KW, "keys per warp");
        constexpr int LPK = DH / 16;      // lanes per key row: 16 or 8
        constexpr int KPI = 32 / LPK;     // keys per copy instruction: 2 or 4
        const bool kg = warp < KW;
        const int kbase = (warp % KW) * KPW;
        const int ul = lane % LPK;        // lane covers bytes 16 ul .. 16 ul + 15
        const uint8_t* cache = kg ? P.kcache8 : P.vcache8;
        uint32_t g = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < NU && ok; u += P.G) {
            const int nt = unit_tiles<PAIR>(P, u);
            for (int t = 0; t < nt && ok; ++t, ++g) {
                const int slot = (int)(g % NI);
                if (!mbar_wait(bar(F_IFULL + slot), (g / NI) & 1, abort_flag, P.err)) {
                    ok = false;
                    break;
                }
                const int tok1 = idx[slot * TILE + kbase + lane];
                mbar_arrive(bar(F_IEMPTY + slot));
                const size_t row1 = tok1 >= 0 ? (size_t)tok1 * tok_stride : 0;
                uint32_t tile, fullb;
                if (kg) {
                    const int kb = (int)(g % F8_NKB);
                    if (!mbar_wait(bar(F_KEMPTY + kb), ((g / F8_NKB) & 1) ^ 1, abort_flag, P.err)) {
                        ok = false;
                        break;
                    }
                    tile = sbase + L::OFF_K + kb * RAW_TILE;
                    fullb = bar(F_KFULL + kb);
                } else {
                    const int vb = (int)(g % F8_NVB);
                    if (!mbar_wait(bar(F_VEMPTY + vb), ((g / F8_NVB) & 1) ^ 1, abort_flag, P.err)) {
                        ok = false;
                        break;
                    }
                    tile = sbase + L::OFF_V + vb * RAW_TILE;
                    fullb = bar(F_VFULL + vb);
                }
#pragma unroll 4
                for (int e = 0; e < KPW / KPI; ++e) {
                    const int src = KPI * e + lane / LPK;   // lane holding this key's row
                    const int key = kbase + src;
                    const int tok = __shfl_sync(0xffffffffu, tok1, src);
                    const size_t row = __shfl_sync(0xffffffffu, row1, src);
                    // half ul / 8, unit ul % 8 of the key's swizzled row
                    const uint32_t dst = tile + (ul >> 3) * (TILE * 128) + sw128(key, ul & 7);
                    const uint8_t* sp = tok >= 0 ? cache + row + ul * 16 : cache;
                    cp_async16(dst, sp, tok >= 0 ? 16u : 0u);
                }
                cp_async_arrive(fullb);
            }
        }
        if (!ok) asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------------------ UMMA issuer
        // Per row: Q.K^T(g), then P.V(g - 1) once its P is ready; the row's
        // last P.V before the next row's first Q.K^T.
        if (lane == 0) {
            bool ok = true;
            auto issue_pv = [&](uint32_t x, bool first) -> bool {
                if (!mbar_wait(bar(F_PREADY + (x & 1)), (x >> 1) & 1, abort_flag, P.err))
                    return false;
                const int vb = (int)(x % F8_NVB);
                if (!mbar_wait(bar(F_VFULL + vb), (x / F8_NVB) & 1, abort_flag, P.err)) return false;
                // cp.async writes are generic-proxy writes; order them before UMMA reads.
                fence_async_shared();
                tc_fence_after();
                const uint32_t vst = sbase + L::OFF_V + vb * RAW_TILE;
                const uint32_t pt = sbase + L::OFF_PT + (x & 1) * L::PT_BYTES;
#pragma unroll
                for (int h = 0; h < HALVES; ++h) {
#pragma unroll
                    for (int ks = 0; ks < TILE / 32; ++ks) {
                        // V^T half h: M = 128 d (one 128-byte atom), K = 32 keys (rows)
                        const uint64_t a = sdesc_sw128(vst + h * (TILE * 128) + ks * 4096, TILE * 128, 1024);
                        const uint64_t b = sdesc_sw128(pt + ks * 32, 16, 1024);
                        umma_f8(tmem + L::O_COL + h * N3, a, b, IDESC_PV, (!first || ks > 0));
                    }
                }
                umma_commit(bar(F_PTEMPTY + (x & 1)));
                umma_commit(bar(F_VEMPTY + vb));
                return true;
            };
            uint32_t g = 0;
            int rloc = 0;
            for (int u = blockIdx.x; u < NU && ok; u += P.G) {
                const int nt = unit_tiles<PAIR>(P, u);
                if (nt == 0) continue;
                const int qb = rloc % F8_NQB;
                if (!mbar_wait(bar(F_QFULL + qb), (rloc / F8_NQB) & 1, abort_flag, P.err)) {
                    ok = false;
                    break;
                }
                ++rloc;
                const uint32_t sq = sbase + L::OFF_Q + qb * L::Q_BYTES;
                const uint32_t g0 = g;
                for (int t = 0; t < nt; ++t, ++g) {
                    const int kb = (int)(g % F8_NKB);
                    if (!mbar_wait(bar(F_KFULL + kb), (g / F8_NKB) & 1, abort_flag, P.err)) {
                        ok = false;
                        break;
                    }
                    fence_async_shared();
                    tc_fence_after();
                    const uint32_t kst = sbase + L::OFF_K + kb * RAW_TILE;
#pragma unroll
                    for (int kk = 0; kk < DH / 32; ++kk) {
                        const int h = kk >> 2;   // d half
                        const uint64_t a = sdesc_sw128(kst + h * (TILE * 128) + (kk & 3) * 32, 16, 1024);
                        const uint64_t b = sdesc_sw128(sq + h * (N3 * 128) + (kk & 3) * 32, 16, 1024);
                        umma_f8(tmem + L::S_COL + (g & 1) * N3, a, b, IDESC_QK, kk > 0);
                    }
                    umma_commit(bar(F_SFULL + (g & 1)));
                    umma_commit(bar(F_KEMPTY + kb));
                    if (t == nt - 1) umma_commit(bar(F_QEMPTY + qb));
                    if (t >= 1 && !(ok = issue_pv(g - 1, g - 1 == g0))) break;
                }
                if (ok) ok = issue_pv(g - 1, g - 1 == g0);
            }
            if (!ok) {
                umma_commit(bar(F_DRAIN));
                drain_wait(bar(F_DRAIN), 0);
            }
        }
    } else if (warp < KEY_WARP0 + 4) {
        // ------------------------------------------------------------ key warps
        // Each thread keeps every head's reference max in registers: after a
        // vote fires, the warps' partial maxima go through shared memory and
        // one barrier, and every thread derives the same new references.
        const int wq = warp & 3;
        const int k = wq * 32 + lane;
        const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
        // The keys are the codes' values: the K scale joins the score scale.
        const float sl2k = P.scale_log2 * __ldg(P.kscale);
        const float vsc = __ldg(P.vscale);
        // P^T row r, key k: byte r * 128 + (((k >> 4) ^ (r & 7)) << 4) + (k & 15).
        const uint32_t p_key = (uint32_t)k & 15u, p_unit = (uint32_t)k >> 4;
        auto pofs = [&](int r) -> uint32_t {
            return (uint32_t)r * 128u + ((p_unit ^ ((uint32_t)r & 7u)) << 4) + p_key;
        };
        uint32_t g = 0;
        uint32_t gphase = 0;
        int rloc = 0;
        bool ok = true;
        if constexpr (PAIR) {
            // Units of two rows, one tile each: S^T column c is head c & 7 of
            // row 2u + (c >> 3); key k belongs to row 2u + (k >> 6).
            for (int u = blockIdx.x; u < NU && ok; u += P.G) {
                const int i0 = 2 * u;
                if (unit_tiles<PAIR>(P, u) == 0) {
                    // Nothing selected in either row: both outputs are zero.
                    for (int sr = 0; sr < 2 && i0 + sr < P.rows; ++sr)
                        for (int v = k; v < HQ * (DH / 8); v += 128)
                            reinterpret_cast<uint4*>(P.out + (size_t)(i0 + sr) * q_stride)[v] =
                                make_uint4(0, 0, 0, 0);
                    continue;
                }
                const int qb = rloc % F8_NQB;
                ok = mbar_wait(bar(F_QFULL + qb), (rloc / F8_NQB) & 1, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                ++rloc;
                float sl2[NP];
#pragma unroll
                for (int c = 0; c < NP; ++c) sl2[c] = (c & 7) < HQ ? sl2k * qs[qb * NP + c] : 0.f;
                const int b = g & 1;
                bool masked;
                {
                    // The index warp's verdict on this key (-1: masked).
                    const int slot = (int)(g % NI);
                    ok = mbar_wait(bar(F_IFULL + slot), (g / NI) & 1, abort_flag, P.err);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    masked = reinterpret_cast<const int*>(gbase + L::OFF_IDX)[slot * TILE + k] < 0;
                    mbar_arrive(bar(F_IEMPTY + slot));
                }
                ok = mbar_wait(bar(F_SFULL + b), (g >> 1) & 1, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                const int kr = k >> 6;   // the unit's row this key belongs to
                float s[NP];
                {
                    uint32_t r1[TS], r2[TS], r3[TS];
                    const uint32_t sc = t_lane + L::S_COL + b * N3;
                    tmem_ldn<TS>(sc, r1);
                    tmem_ldn<TS>(sc + TS, r2);
                    tmem_ldn<TS>(sc + 2 * TS, r3);
                    tmem_ld_wait<TS>(r1);
                    tmem_ld_wait<TS>(r2);
                    tmem_ld_wait<TS>(r3);
#pragma unroll
                    for (int c = 0; c < NP; ++c)
                        s[c] = (masked || (c >> 3) != kr || (c & 7) >= HQ)
                                   ? -INFINITY
                                   : combine3(r1[c], r2[c], r3[c]) * sl2[c];
                }
                // The unit's one tile: each column's exact max, the reference
                // REF_SHIFT below it.
                float* rd = red + (g & 1) * (4 * NP);
#pragma unroll
                for (int c = 0; c < NP; ++c) {
                    if ((c & 7) >= HQ) continue;
                    float m = s[c];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                    if (lane == 0) rd[wq * NP + c] = m;
                }
                ok = group_sync(bar(F_GROUP), gphase, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                float mr[NP];
#pragma unroll
                for (int c = 0; c < NP; ++c) {
                    const float tmax = fmaxf(fmaxf(rd[c], rd[NP + c]), fmaxf(rd[2 * NP + c], rd[3 * NP + c]));
                    mr[c] = ((c & 7) >= HQ || tmax == -INFINITY) ? 0.f : tmax - REF_SHIFT;
                }
                // P^T buffer b is free once the P.V two tiles back has completed.
                ok = mbar_wait(bar(F_PTEMPTY + b), ((g >> 1) & 1) ^ 1, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                float pl[NP];
                {
                    uint8_t* pt = gbase + L::OFF_PT + b * L::PT_BYTES;
#pragma unroll
                    for (int c = 0; c < NP; c += 2) {
                        pl[c] = pl[c + 1] = 0.f;
                        if ((c & 7) >= HQ) continue;
                        pl[c] = ex2(s[c] - mr[c]);
                        pl[c + 1] = (c & 7) + 1 < HQ ? ex2(s[c + 1] - mr[c + 1]) : 0.f;
                        uint32_t t3[3];
                        split3_e4m3x2(pl[c], pl[c + 1], t3[0], t3[1], t3[2]);
#pragma unroll
                        for (int e = 0; e < 3; ++e) {
                            pt[pofs(e * TS + c)] = (uint8_t)(t3[e] & 0xFF);
                            pt[pofs(e * TS + c + 1)] = (uint8_t)(t3[e] >> 8);
                        }
                    }
                }
                fence_async_shared();
                mbar_arrive(bar(F_PREADY + b));
                // Row sums per column (this tile is the unit's only one), while
                // the P.V runs: warp sums -> redl (slot of this unit's parity).
                float* rl = redl + (rloc & 1) * (4 * NP);
#pragma unroll
                for (int c = 0; c < NP; ++c) {
                    if ((c & 7) >= HQ) continue;
                    float v = pl[c];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == 0) rl[wq * NP + c] = v;
                }
                // ---------------------------------------------------------- unit epilogue
                const uint32_t x = g++;
                ok = mbar_wait(bar(F_PTEMPTY + (x & 1)), (x >> 1) & 1, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                ok = group_sync(bar(F_GROUP), gphase, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                // Every thread has read the unit's Q scales: the buffer may be refilled.
                if (k == 0) mbar_arrive(bar(F_QEMPTY + qb));
                float inv[NP];
#pragma unroll
                for (int c = 0; c < NP; ++c) {
                    const float l = (rl[c] + rl[NP + c]) + (rl[2 * NP + c] + rl[3 * NP + c]);
                    inv[c] = ((c & 7) < HQ && l > 0.f) ? vsc / l : 0.f;
                }
#pragma unroll
                for (int h = 0; h < HALVES; ++h) {
                    uint32_t r1[TS], r2[TS], r3[TS];
                    const uint32_t oc = t_lane + L::O_COL + h * N3;
                    tmem_ldn<TS>(oc, r1);
                    tmem_ldn<TS>(oc + TS, r2);
                    tmem_ldn<TS>(oc + 2 * TS, r3);
                    tmem_ld_wait<TS>(r1);
                    tmem_ld_wait<TS>(r2);
                    tmem_ld_wait<TS>(r3);
                    const int d = h * 128 + k;
#pragma unroll
                    for (int c = 0; c < NP; ++c) {
                        const int row = i0 + (c >> 3);
                        if ((c & 7) < HQ && row < P.rows)
                            P.out[(size_t)row * q_stride + (c & 7) * DH + d] =
                                __float2half_rn(combine3(r1[c], r2[c], r3[c]) * inv[c]);
                    }
                }
            }
        } else {
            for (int u = blockIdx.x; u < NU && ok; u += P.G) {
                const int nt = unit_tiles<PAIR>(P, u);
                const int i = u;   // the row (without PAIR)
                if (nt == 0) {
                    // Nothing selected: the row's output is zero.
                    for (int u = k; u < nh * (DH / 8); u += 128)
                        reinterpret_cast<uint4*>(P.out + (size_t)i * q_stride)[u] = make_uint4(0, 0, 0, 0);
                    continue;
                }
                const int qb = rloc % F8_NQB;
                ok = mbar_wait(bar(F_QFULL + qb), (rloc / F8_NQB) & 1, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                ++rloc;
                // Score scale per head (log2 units): scale * kscale * the head's Q scale.
                float sl2[HQ], mr[HQ], lpart[HQ];
    #pragma unroll
                for (int c = 0; c < HQ; ++c) {
                    sl2[c] = c < nh ? sl2k * qs[qb * NP + c] : 0.f;
                    mr[c] = -INFINITY;
                    lpart[c] = 0.f;
                }
                for (int t = 0; t < nt; ++t, ++g) {
                    const int b = g & 1;
                    bool masked;
                    {
                        // The index warp's verdict on this key (-1: masked).
                        const int slot = (int)(g % NI);
                        ok = mbar_wait(bar(F_IFULL + slot), (g / NI) & 1, abort_flag, P.err);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                        masked = reinterpret_cast<const int*>(gbase + L::OFF_IDX)[slot * TILE + k] < 0;
                        mbar_arrive(bar(F_IEMPTY + slot));
                    }
                    ok = mbar_wait(bar(F_SFULL + b), (g >> 1) & 1, abort_flag, P.err);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after();
                    float s[HQ];
                    {
                        uint32_t r1[TS], r2[TS], r3[TS];
                        const uint32_t sc = t_lane + L::S_COL + b * N3;
                        tmem_ldn<TS>(sc, r1);
                        tmem_ldn<TS>(sc + TS, r2);
                        tmem_ldn<TS>(sc + 2 * TS, r3);
                        tmem_ld_wait<TS>(r1);
                        tmem_ld_wait<TS>(r2);
                        tmem_ld_wait<TS>(r3);
    #pragma unroll
                        for (int c = 0; c < HQ; ++c)
                            s[c] = masked ? -INFINITY : combine3(r1[c], r2[c], r3[c]) * sl2[c];
                    }
                    // A row's first tile always takes the exact max (its references
                    // are -inf); later tiles only when a score crosses its reference.
                    bool any = t == 0;
                    if (!any) {
                        bool exceed = false;
    #pragma unroll
                        for (int c = 0; c < HQ; ++c)
                            if (c < nh) exceed |= s[c] > mr[c] + RESCALE_THRESHOLD;
                        const unsigned vote = __ballot_sync(0xffffffffu, exceed);
                        volatile int* fl = flags + (g & 1) * 4;
                        if (lane == 0) fl[wq] = vote != 0;
                        ok = group_sync(bar(F_GROUP), gphase, abort_flag, P.err);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                        any = fl[0] | fl[1] | fl[2] | fl[3];
                    }
                    if (any) {
                        // The tile's max per head: warp maxima -> red (its slot of
                        // this tile parity) -> one barrier -> every thread.
                        float* rd = red + (g & 1) * (4 * NP);
    #pragma unroll
                        for (int c = 0; c < HQ; ++c) {
                            if (c >= nh) break;
                            float m = s[c];
    #pragma unroll
                            for (int o = 16; o > 0; o >>= 1)
                                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                            if (lane == 0) rd[wq * NP + c] = m;
                        }
                        ok = group_sync(bar(F_GROUP), gphase, abort_flag, P.err);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                        float f[HQ];
    #pragma unroll
                        for (int c = 0; c < HQ; ++c) {
                            f[c] = 1.0f;
                            if (c < nh) {
                                const float tmax = fmaxf(fmaxf(rd[c], rd[NP + c]),
                                                         fmaxf(rd[2 * NP + c], rd[3 * NP + c]));
                                if (tmax > mr[c] + RESCALE_THRESHOLD) {
                                    const float ref = tmax - REF_SHIFT;
                                    f[c] = (mr[c] == -INFINITY) ? 0.f : ex2(mr[c] - ref);
                                    mr[c] = ref;
                                }
                            }
                        }
                        if (t > 0) {
                            // O^T must hold every earlier P.V of the row before it is rescaled.
                            const uint32_t x = g - 1;
                            ok = mbar_wait(bar(F_PTEMPTY + (x & 1)), (x >> 1) & 1, abort_flag, P.err);
                            ok = __all_sync(0xffffffffu, ok);
                            if (!ok) break;
                            tc_fence_after();
    #pragma unroll
                            for (int g6 = 0; g6 < 3 * HALVES; ++g6) {   // (d half, expansion term)
                                const uint32_t col = L::O_COL + (g6 / 3) * N3 + (g6 % 3) * TS;
                                uint32_t r[TS];
                                tmem_ldn<TS>(t_lane + col, r);
                                tmem_ld_wait<TS>(r);
    #pragma unroll
                                for (int c = 0; c < HQ; ++c)
                                    r[c] = __float_as_uint(__uint_as_float(r[c]) * f[c]);
                                tmem_stn<TS>(t_lane + col, r);
                            }
                            tmem_st_wait();
                        }
    #pragma unroll
                        for (int c = 0; c < HQ; ++c) lpart[c] *= f[c];
                    }
                    // P^T buffer b is free once the P.V two tiles back has completed.
                    ok = mbar_wait(bar(F_PTEMPTY + b), ((g >> 1) & 1) ^ 1, abort_flag, P.err);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    {
                        // [P1 | P2 | P3]^T, K-major: row = term * TS + head, byte = key.
                        uint8_t* pt = gbase + L::OFF_PT + b * L::PT_BYTES;
    #pragma unroll
                        for (int c = 0; c < HQ; c += 2) {
                            if (c >= nh) break;
                            const float p0 = ex2(s[c] - (mr[c] == -INFINITY ? 0.f : mr[c]));
                            const float p1 = c + 1 < nh ? ex2(s[c + 1] - (mr[c + 1] == -INFINITY ? 0.f : mr[c + 1]))
                                                        : 0.f;
                            lpart[c] += p0;
                            lpart[c + 1] += p1;
                            uint32_t t3[3];
                            split3_e4m3x2(p0, p1, t3[0], t3[1], t3[2]);
    #pragma unroll
                            for (int e = 0; e < 3; ++e) {
                                pt[pofs(e * TS + c)] = (uint8_t)(t3[e] & 0xFF);
                                pt[pofs(e * TS + c + 1)] = (uint8_t)(t3[e] >> 8);
                            }
                        }
                    }
                    fence_async_shared();
                    mbar_arrive(bar(F_PREADY + b));
                }
                if (!ok) break;
                // ---------------------------------------------------------- row epilogue
                const uint32_t x = g - 1;
                ok = mbar_wait(bar(F_PTEMPTY + (x & 1)), (x >> 1) & 1, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                // Row sums: warp sums -> redl (its slot of this row parity) -> one
                // barrier.  The next write to the same slot comes two rows later,
                // behind barriers every thread passes after its reads here.
                float* rl = redl + (rloc & 1) * (4 * NP);
    #pragma unroll
                for (int c = 0; c < HQ; ++c) {
                    if (c >= nh) break;
                    float v = lpart[c];
    #pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == 0) rl[wq * NP + c] = v;
                }
                ok = group_sync(bar(F_GROUP), gphase, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                // Every thread has read this row's Q scales (row start) and passed
                // the barrier above: the Q buffer may be refilled.
                if (k == 0) mbar_arrive(bar(F_QEMPTY + qb));
                float inv[HQ];
    #pragma unroll
                for (int c = 0; c < HQ; ++c) {
                    const float l = (rl[c] + rl[NP + c]) + (rl[2 * NP + c] + rl[3 * NP + c]);
                    inv[c] = l > 0.f ? vsc / l : 0.f;
                }
    #pragma unroll
                for (int h = 0; h < HALVES; ++h) {
                    uint32_t r1[TS], r2[TS], r3[TS];
                    const uint32_t oc = t_lane + L::O_COL + h * N3;
                    tmem_ldn<TS>(oc, r1);
                    tmem_ldn<TS>(oc + TS, r2);
                    tmem_ldn<TS>(oc + 2 * TS, r3);
                    tmem_ld_wait<TS>(r1);
                    tmem_ld_wait<TS>(r2);
                    tmem_ld_wait<TS>(r3);
                    const int d = h * 128 + k;
    #pragma unroll
                    for (int c = 0; c < HQ; ++c)
                        if (c < nh)
                            P.out[(size_t)i * q_stride + c * DH + d] =
                                __float2half_rn(combine3(r1[c], r2[c], r3[c]) * inv[c]);
                }
            }
        }
    } else if (warp == IDX_WARP) {
        if constexpr (PAIR)
            index_warp_pairs(P, reinterpret_cast<int*>(gbase + L::OFF_IDX), bar(F_IFULL),
                             bar(F_IEMPTY), abort_flag);
        else
            index_warp(P, reinterpret_cast<int*>(gbase + L::OFF_IDX),
                       reinterpret_cast<uint32_t*>(gbase + L::OFF_SEEN), bar(F_IFULL),
                       bar(F_IEMPTY), abort_flag);
    } else {
        // ------------------------------------------------------------ Q expansion
        // A unit's head rows (its row's heads, or with PAIR both rows' heads,
        // entry e = row * HQ + head) are dealt to the warps: warp qw takes
        // entries qw, qw + F8_QWARPS, ...  Each lane loads EPL values of an
        // entry's head row (all of the unit's loads issued before the wait
        // for the buffer), the head's scale is its absolute max / 256, and the
        // three E4M3 terms of x / scale go to rows col, TS + col and 2 TS + col
        // of the K-major, 128B-swizzled expansion (col: the head's S^T column).
        const int qw = warp - Q_WARP0;
        constexpr int NE_MAX = PAIR ? 2 * HQ : HQ;
        const int ne = PAIR ? 2 * HQ : nh;
        constexpr int RPW = (NE_MAX + F8_QWARPS - 1) / F8_QWARPS;
        constexpr int EPL = DH / 32;   // elements of a row per lane: 8 or 4
        using QV = typename std::conditional<EPL == 8, uint4, uint2>::type;
        const int d0 = lane * EPL;
        int rloc = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < NU && ok; u += P.G) {
            const int nt = unit_tiles<PAIR>(P, u);
            if (nt == 0) continue;
            const int qb = rloc % F8_NQB;
            // Entry e: row, head and S^T column.
            auto entry = [&](int e, int& row, int& head, int& col) {
                const int sr = PAIR ? e / HQ : 0;
                head = e - sr * HQ;
                row = PAIR ? 2 * u + sr : u;
                col = sr * 8 + head;
            };
            QV raw[RPW];
#pragma unroll
            for (int j = 0; j < RPW; ++j) {
                const int e = qw + F8_QWARPS * j;
                int row, head, col;
                entry(e, row, head, col);
                raw[j] = (e < ne && row < P.rows)
                             ? *reinterpret_cast<const QV*>(P.q + (size_t)row * q_stride + head * DH + d0)
                             : QV{};
            }
            ok = mbar_wait(bar(F_QEMPTY + qb), ((rloc / F8_NQB) & 1) ^ 1, abort_flag, P.err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            uint8_t* qbuf = gbase + L::OFF_Q + qb * L::Q_BYTES;
#pragma unroll
            for (int j = 0; j < RPW; ++j) {
                const int e = qw + F8_QWARPS * j;
                if (e >= ne) break;
                int row, head, c;
                entry(e, row, head, c);
                if (row >= P.rows) continue;   // the missing second row of the last unit
                float x[EPL];
                const __half* hx = reinterpret_cast<const __half*>(&raw[j]);
#pragma unroll
                for (int e = 0; e < EPL; ++e) x[e] = __half2float(hx[e]);
                float amax = 0.f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                const float sc = amax > 0.f ? amax / 256.0f : 1.0f;
                const float inv = 1.0f / sc;
                uint32_t w1[2] = {0, 0}, w2[2] = {0, 0}, w3[2] = {0, 0};
#pragma unroll
                for (int e = 0; e < EPL; e += 2) {
                    uint32_t b1, b2, b3;
                    split3_e4m3x2(x[e] * inv, x[e + 1] * inv, b1, b2, b3);
                    w1[e >> 2] |= b1 << (8 * (e & 3));
                    w2[e >> 2] |= b2 << (8 * (e & 3));
                    w3[e >> 2] |= b3 << (8 * (e & 3));
                }
                const int h = d0 >> 7, cin = d0 & 127;
                uint8_t* qh = qbuf + h * (N3 * 128) + (cin & 15);
                if constexpr (EPL == 8) {
                    *reinterpret_cast<uint2*>(qh + sw128(c, cin >> 4)) = make_uint2(w1[0], w1[1]);
                    *reinterpret_cast<uint2*>(qh + sw128(TS + c, cin >> 4)) = make_uint2(w2[0], w2[1]);
                    *reinterpret_cast<uint2*>(qh + sw128(2 * TS + c, cin >> 4)) = make_uint2(w3[0], w3[1]);
                } else {
                    *reinterpret_cast<uint32_t*>(qh + sw128(c, cin >> 4)) = w1[0];
                    *reinterpret_cast<uint32_t*>(qh + sw128(TS + c, cin >> 4)) = w2[0];
                    *reinterpret_cast<uint32_t*>(qh + sw128(2 * TS + c, cin >> 4)) = w3[0];
                }
                if (lane == 0) qs[qb * NP + c] = sc;
            }
            // Generic-proxy stores, read by the tensor cores (async proxy).
            fence_async_shared();
            mbar_arrive(bar(F_QFULL + qb));
            ++rloc;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, F8_TMEM_COLS);
    }
}

}  // namespace sparse

int sparse_launch(const void* q, const void* kcache, const void* vcache, const float* kscale,
                  const float* vscale, bool e4m3, const int32_t* block_table,
                  const int32_t* sel_idx, const int32_t* sel_cnt, int max_sel, int num_pages,
                  int page, int ctx_len, int rows, int Hq, int Hkv, int Dh, float scale,
                  void* out, cudaStream_t stream) {
    using namespace sparse;
    const DeviceInfo* di = device_info();
    if (!di) return GQA_ERR_CUDA;
    const int grp = Hq / Hkv;
    Params P;
    P.table = block_table;
    P.sel_idx = sel_idx;
    P.sel_cnt = sel_cnt;
    P.max_sel = max_sel;
    P.num_pages = num_pages;
    P.log2_page = __builtin_ctz((unsigned)page);
    P.ctx_len = ctx_len;
    P.rows = rows;
    P.G = rows < di->num_sms ? rows : di->num_sms;
    P.nh = grp;
    P.q_stride = Hq * Dh;
    P.kv_stride = Hkv * Dh;
    P.kscale = kscale;
    P.vscale = vscale;
    P.scale_log2 = scale * 1.4426950408889634f;
    P.err = di->err_word;
    // The 6-head instantiations address the caches with a stride of one head,
    // so they serve one KV head only.
    const bool six = (grp == kHq && Hkv == 1);
    using KernelFn = void (*)(Params);
    KernelFn fn;
    int smem, threads;
    if (e4m3) {
        // The 6-head family takes two rows per tile when every row's selection
        // fits half a tile (at most 64 keys); the grid then walks row pairs.
        const bool pair = six && max_sel * BLK <= TILE / 2;
        if (pair) {
            const int units = (rows + 1) / 2;
            P.G = units < di->num_sms ? units : di->num_sms;
        }
        if (Dh == 128) {
            fn = pair ? sparse_f8_kernel<kHq, 128, true>
                      : (six ? sparse_f8_kernel<kHq, 128, false> : sparse_f8_kernel<NP, 128, false>);
            threads = pair ? f8_nthreads<kHq, 128, true>()
                           : (six ? f8_nthreads<kHq, 128, false>() : f8_nthreads<NP, 128, false>());
            smem = pair ? SL8<kHq, 128, true>::SMEM
                        : (six ? SL8<kHq, 128, false>::SMEM : SL8<NP, 128, false>::SMEM);
        } else {
            fn = pair ? sparse_f8_kernel<kHq, 256, true>
                      : (six ? sparse_f8_kernel<kHq, 256, false> : sparse_f8_kernel<NP, 256, false>);
            threads = pair ? f8_nthreads<kHq, 256, true>()
                           : (six ? f8_nthreads<kHq, 256, false>() : f8_nthreads<NP, 256, false>());
            smem = pair ? SL8<kHq, 256, true>::SMEM
                        : (six ? SL8<kHq, 256, false>::SMEM : SL8<NP, 256, false>::SMEM);
        }
    } else {
        // As above: two rows per tile for the 6-head family when they fit.
        const bool pair = six && max_sel * BLK <= TILE / 2;
        if (pair) {
            const int units = (rows + 1) / 2;
            P.G = units < di->num_sms ? units : di->num_sms;
        }
        if (Dh == 128) {
            fn = pair ? sparse_kernel<kHq, 128, true>
                      : (six ? sparse_kernel<kHq, 128, false> : sparse_kernel<NP, 128, false>);
            threads = six ? nthreads<kHq, 128>() : nthreads<NP, 128>();
            smem = smem_bytes<128>();
        } else {
            fn = pair ? sparse_kernel<kHq, 256, true>
                      : (six ? sparse_kernel<kHq, 256, false> : sparse_kernel<NP, 256, false>);
            threads = six ? nthreads<kHq, 256>() : nthreads<NP, 256>();
            smem = smem_bytes<256>();
        }
    }
    if (ensure_smem_limit(reinterpret_cast<const void*>(fn), smem) != GQA_OK)
        return GQA_ERR_CUDA;
    // One launch per KV head: query heads g * grp .. g * grp + grp - 1 read
    // token rows of KV head g.
    const size_t esz = e4m3 ? 1 : 2;   // bytes per cache element
    for (int g = 0; g < Hkv; ++g) {
        P.q = static_cast<const __half*>(q) + (size_t)g * grp * Dh;
        P.out = static_cast<__half*>(out) + (size_t)g * grp * Dh;
        const uint8_t* kb = static_cast<const uint8_t*>(kcache) + (size_t)g * Dh * esz;
        const uint8_t* vb = static_cast<const uint8_t*>(vcache) + (size_t)g * Dh * esz;
        P.kcache = reinterpret_cast<const __half*>(kb);
        P.vcache = reinterpret_cast<const __half*>(vb);
        P.kcache8 = kb;
        P.vcache8 = vb;
        fn<<<P.G, threads, smem, stream>>>(P);
        if (cudaGetLastError() != cudaSuccess) return GQA_ERR_CUDA;
    }
    return GQA_OK;
}

}  // namespace gqa
