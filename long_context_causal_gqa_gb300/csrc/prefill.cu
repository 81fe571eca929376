// prefill.cu -- dense causal GQA prefill on sm_103a.
//
// Problem ("[Kernel][SM70] Default long-prefill GQA architecture", Purpose):
// q [Q, 6, 256], k/v [KV, 1, 256] fp16, scale 1/16, query row i bottom-right
// aligned (sees keys 0 .. KV - Q + i), fp16 output.  The page packs the six
// query heads that share the KV head into wide QK / PV GEMMs and merges the
// causal tail with online-softmax state; both ideas carry over, re-shaped for
// tcgen05:
//
// * Head packing.  q is [Q, 6, 256] = [6Q, 256] row-major, so consecutive
//   flattened rows (positions x 6 heads) form the M tiles with no padding.
//   Other groupings at D = 256: with one KV head and Hq query heads the
//   packed rows are positions x Hq; with Hkv > 1 KV heads every query head
//   has its own pair tiles (one packed row per position) in the same launch,
//   reading the KV head h / (Hq / Hkv) through 3-D tensor maps
//   (d, head, row).
// * CTA pairs (cta_group::2).  A cluster of two CTAs on neighbouring SMs
//   takes a pair tile of 256 packed rows, 128 per CTA, and runs one M = 256
//   UMMA stream issued by the even CTA:
//     S[256 x 128 keys]  = Q[256 x 256] . K^T     (K-major operands)
//     O[256 x 256 d]    += P[256 x 128] . V        (P from tensor memory)
//   Each CTA holds its own 128 rows of Q, S, P and O, but only half of every
//   K tile (64 keys) and half of every V tile (128 of the 256 d), so a K/V
//   tile costs each SM 64 KB of shared-memory traffic instead of 128 KB and
//   the copy ring covers twice as many tiles of L2 latency.
// * Warp roles per CTA: warp 0 loads Q and K, warp 10 loads V (each its
//   half of every operand; the odd CTA's copies complete on the even CTA's
//   barriers), warp 1 tensor-memory owner and, in the even CTA, the thread
//   that issues the UMMAs, warps 2..9 softmax + epilogue in two warpgroups,
//   each thread one tile row (TMEM lane) and half of its columns.  At head
//   size 128 one more warp's first thread (even CTA) issues every P.V while
//   warp 1 issues every Q.K^T (see the issuer section).
// * K and V stream through separate rings of 16 KB slots, so that K of the
//   next tiles never waits behind V slots held until their P is ready.  With
//   fp16 K / V each ring holds one tile per S buffer: a tile's K slots are
//   refilled after the Q.K^T into the same-numbered S buffer completes and
//   its V slots after that tile's P.V does, signalled by the scores-ready and
//   O-ready barriers the softmax waits on anyway, so the issuing thread
//   commits no per-slot releases and takes one barrier per tile and operand
//   (with one issuing thread, half of each tile's issue time had been
//   barrier operations).
// * Tensor memory (512 columns x 128 lanes per CTA): O = DH fp32 columns,
//   then two (DH = 256) or three (DH = 128) S buffers of 128 fp32 columns, so
//   Q.K^T of tile j+1 runs while tile j's softmax runs.  Each warpgroup's P (fp16) overwrites the first 32
//   columns of its own 64-column half of the S buffer.  The two threads of a
//   row swap their half maxima through shared memory each tile, so both take
//   the same rescale decisions.
// * Online softmax with a lazy rescale: the per-row reference max only moves
//   (and O is rescaled in TMEM) when a tile's max exceeds it by more than
//   8 (log2 units), which bounds P by 256.
// * Only the one or two KV tiles on a pair tile's diagonal are masked.
// * Work split: the causal-visible (pair tile, kv tile) iterations are laid
//   out pair-tile-major and cut into one contiguous, equal range per CTA pair
//   (shape-only, so deterministic).  A pair tile cut between pairs leaves
//   (O, m, l) partials in the workspace; a merge kernel combines them in pair
//   order (exact log-sum-exp merge).
#include <atomic>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"
#include "sm100.cuh"

namespace gqa {
namespace prefill {

constexpr int BM = 128;         // packed query rows per CTA
constexpr int BM2 = 2 * BM;     // packed query rows per CTA pair
constexpr int BN = 128;         // keys per KV tile
constexpr int D = kHeadDim;     // 256, the largest head size; shared memory is laid out for it
// Ring slots of 16 KB.  A K slot holds this CTA's 64 keys x two 64-wide d
// chunks (8 KB each); a V slot holds 32-key sub-tiles x this CTA's DH / 2 d
// (64-wide atoms of 4 KB: two sub-tiles of two atoms at DH = 256, four of
// one at DH = 128).  A tile's half of K or V is DH / 128 slots.
constexpr int SLOT_BYTES = 16384;
constexpr int HALF_SLOT = SLOT_BYTES / 2;
constexpr int Q_BYTES = BM * D * 2;           // 64 KB (the DH = 256 Q tile)
constexpr int NWG = 2;                        // softmax warpgroups per CTA
constexpr int COLS = BN / NWG;                // S columns per softmax thread
constexpr int NSOFT = 128 * NWG;              // softmax threads per CTA
constexpr int V_WARP = 2 + NSOFT / 32;
constexpr int XCH_BYTES = 3 * NWG * BM * 4;  // part maxima [parity][part][row], sums [part][row]

// S buffers follow O in tensor memory: two of 128 columns after a 256-column
// O (DH = 256), three after a 128-column O (DH = 128).
template <int DH>
struct SBuf {
    static constexpr int N = DH == 128 ? 3 : 2;
    static constexpr uint32_t COL0 = DH;
};

// Per-variant sizes.  fp16 K / V: the K and V rings hold one tile per S
// buffer (DH / 128 slots each), so a K tile's slots are free again exactly
// when the Q.K^T into the same-numbered S buffer has completed (its
// scores-ready barrier) and a V tile's when the P.V of that tile has (its
// O-ready barrier): no per-slot release barriers or commits.
// F8 (K and V stored as FP8-E4M3 codes): four converter warps (two for K,
// two for V, each half of a slot's rows) load each CTA's codes of a tile from
// global memory into registers and write them as fp16 into the same ring
// slots, released the same way.  Up to 16 warps share the same register
// limit (128 per thread at 4 warps per scheduler), so the converters cost no
// registers beyond 13 warps.
// Barriers: ring full/empty (empty: unused), q full/empty, s / p / o [3],
// drain[2], group.
template <bool F8, int DH>
struct Cfg {
    static constexpr int NK = (DH / 128) * SBuf<DH>::N;   // K slots (DH / 128 per tile)
    static constexpr int NV = (DH / 128) * SBuf<DH>::N;   // V slots (DH / 128 per tile)
    static constexpr int NRING = NK + NV;
    static constexpr int RING_BYTES = NRING * SLOT_BYTES;
    static constexpr int NUM_BARS = 2 * NRING + 14;
    static constexpr int NCONV = F8 ? 4 : 0;              // converter warps: 2 for K, 2 for V
    // DH = 128 (three S buffers): one more warp, whose first thread issues the
    // P.V UMMAs; DH = 256: none (-1).
    static constexpr int PV_WARP = DH == 128 ? V_WARP + 1 + NCONV : -1;
    static constexpr int NTHREADS = 32 * (V_WARP + 1 + NCONV + (DH == 128 ? 1 : 0));
    static constexpr int SMEM_BYTES = 1024 /*align slack*/ + RING_BYTES + Q_BYTES +
                                      XCH_BYTES + NUM_BARS * 8 + 16;
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t O_COL = 0;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units
constexpr int kMaxClusters = 80;

// UMMA shapes (M = 256 over the pair): S[256 x 128] = Q[256 x 16] K^T, both
// K-major; O[256 x DH] += P[256 x 16] (tensor memory) V[16 x DH], V MN-major.
constexpr uint32_t IDESC_QK = idesc_f16_f32(256, 128, false, false);

struct Params {
    int Q, KV, M_total, num_ptiles, G;   // M_total, num_ptiles: per head of the tile space
    int heads;            // heads in the tile space: 1 (packed) or Hq (one per query head)
    int head_group;       // query heads per KV head (maps a head of the tile space to its KV head)
    FastDiv grp;          // packed rows per query position
    int out_stride;       // elements between consecutive packed rows of out
    long long total;      // causal-visible (pair tile, kv tile) iterations
    float scale_log2;     // scale * log2(e)
    const float* kscale;  // E4M3 K / V scales (device, one fp32 each); null for fp16 K / V
    const float* vscale;
    const uint8_t* k8;    // E4M3 K / V codes [KV][Hkv][DH] (F8 only)
    const uint8_t* v8;
    int kv_rs;            // bytes between consecutive keys of k8 / v8 (Hkv * DH)
    __half* out;
    FastDiv ptiles;       // divides a tile-space index by num_ptiles (its head)
    float* ws_o;          // [G][2][BM2][DH] unnormalised partial O
    float* ws_ml;         // [G][2][BM2][2] partial (m in log2 units, l)
    unsigned* err;
};

// KV tiles pair tile t needs: up to the last visible key of its last valid row.
__host__ __device__ inline int kv_tiles(int t, int Q, int KV, int M_total, const FastDiv& grp) {
    int last = min(t * BM2 + BM2 - 1, M_total - 1);
    return (KV - Q + grp.div(last)) / BN + 1;
}

__host__ __device__ inline long long pair_begin(long long total, int G, int c) {
    return (long long)c * total / G;
}

// Walks the segments (pair tile, [jb, je)) of one pair's iteration range.
// The tile space is heads x num_ptiles pair tiles, head-major; t is the index
// in it, (hd, lt) its head and pair tile within the head.  With MH false the
// tile space is one head (packed rows) and hd stays 0.
template <bool MH>
struct SegIter {
    long long pos, end, cum;
    int t, hd, lt;
    bool first;
    __device__ void advance(const Params& P) {
        ++t;
        ++lt;
        if (MH && lt == P.num_ptiles) {
            lt = 0;
            ++hd;
        }
    }
    __device__ void init(const Params& P, int pair) {
        pos = pair_begin(P.total, P.G, pair);
        end = pair_begin(P.total, P.G, pair + 1);
        t = 0;
        hd = 0;
        lt = 0;
        cum = 0;
        first = true;
        const int tiles = MH ? P.heads * P.num_ptiles : P.num_ptiles;
        while (t < tiles) {
            int n = kv_tiles(lt, P.Q, P.KV, P.M_total, P.grp);
            if (cum + n > pos) break;
            cum += n;
            advance(P);
        }
    }
    // Next segment: pair tile pt of head head; is_first tells whether it is
    // this pair's first segment.
    __device__ bool next(const Params& P, int& pt, int& head, int& jb, int& je, int& n,
                         bool& is_first) {
        if (pos >= end) return false;
        n = kv_tiles(lt, P.Q, P.KV, P.M_total, P.grp);
        pt = lt;
        head = hd;
        jb = (int)(pos - cum);
        long long e = end - cum;
        je = e < n ? (int)e : n;
        is_first = first;
        first = false;
        pos = cum + je;
        if (je == n) {
            cum += n;
            advance(P);
        }
        return true;
    }
};

// Barrier addresses for a ring of NR slots (K slots 0 .. NK-1, V slots
// NK .. NR-1).
template <int NR>
struct Bars {
    uint32_t b;
    __device__ uint32_t full(int s) const { return b + 8 * s; }
    __device__ uint32_t empty(int s) const { return b + 8 * (NR + s); }
    __device__ uint32_t qfull() const { return b + 8 * (2 * NR); }
    __device__ uint32_t qempty() const { return b + 8 * (2 * NR + 1); }
    // S buffer i (up to three): scores ready (Q.K^T into it complete), P
    // ready, and O ready (the P.V of the buffer's tile complete, so also its
    // P and, with fp16 K / V, that tile's V slots free again).
    __device__ uint32_t sfull(int i) const { return b + 8 * (2 * NR + 2 + i); }
    __device__ uint32_t pfull(int i) const { return b + 8 * (2 * NR + 5 + i); }
    __device__ uint32_t ofull(int i) const { return b + 8 * (2 * NR + 8 + i); }
    __device__ uint32_t drain() const { return b + 8 * (2 * NR + 11); }
    __device__ uint32_t drain2() const { return b + 8 * (2 * NR + 12); }
    __device__ uint32_t group() const { return b + 8 * (2 * NR + 13); }
};

// ---------------------------------------------------------------- CTA pairs
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
// The address of the same shared-memory object in the pair's even CTA.
__device__ __forceinline__ uint32_t leader_addr(uint32_t a) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(0));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}
// Arrive on an mbarrier of the even CTA (default .release.cta semantics: the
// tensor-memory writes this signals are ordered by tcgen05.wait::st and
// tcgen05.fence::before_thread_sync, not by the arrive; a cluster-scope
// release here costs about a microsecond per tile).
__device__ __forceinline__ void remote_arrive(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair.
// Coordinates (x = d, y = row) of a 2-D map (MH false) or (x = d, head,
// y = row) of a 3-D map (MH true).
template <bool MH>
__device__ __forceinline__ void tma_load_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                              int32_t x, int32_t head, int32_t y) {
    if (MH)
        asm volatile(
            "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::"
            "complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(head), "r"(y), "r"(bar)
            : "memory");
    else
        asm volatile(
            "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::"
            "complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
            : "memory");
}
__device__ __forceinline__ void umma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Shared-memory descriptors split into their two 32-bit words: the high word
// (SBO = 1024, version bit 46, 128-byte swizzle) is the same for every
// operand here; the low word is (address >> 4) | (LBO >> 4) << 16, so an
// operand at a fixed offset from a slot base is one integer add away.
constexpr uint32_t DESC_HI = (1024u >> 4) | (1u << 14) | (2u << 29);
__device__ __forceinline__ uint32_t desc_lo(uint32_t saddr, uint32_t lbo) {
    return (saddr >> 4) | ((lbo >> 4) << 16);
}
__device__ __forceinline__ uint64_t desc64(uint32_t lo) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(DESC_HI));
    return d;
}
// UMMA with a compile-time accumulate flag (no predicate set-up).
template <bool ACC>
__device__ __forceinline__ void umma_ss_pair_c(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc) {
    if constexpr (ACC)
        asm volatile("tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, 1;" ::"r"(d_tmem),
                     "l"(a_desc), "l"(b_desc), "r"(idesc)
                     : "memory");
    else
        asm volatile("tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, 0;" ::"r"(d_tmem),
                     "l"(a_desc), "l"(b_desc), "r"(idesc)
                     : "memory");
}

template <bool ACC>
__device__ __forceinline__ void umma_ts_pair_c(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                               uint32_t idesc) {
    if constexpr (ACC)
        asm volatile("tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, 1;" ::"r"(d_tmem),
                     "r"(a_tmem), "l"(b_desc), "r"(idesc)
                     : "memory");
    else
        asm volatile("tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, 0;" ::"r"(d_tmem),
                     "r"(a_tmem), "l"(b_desc), "r"(idesc)
                     : "memory");
}

// Arrive once on the mbarrier at this offset in both CTAs of the pair when
// every UMMA this thread issued before has completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"((uint16_t)3)
        : "memory");
}

// Bounded wait that ignores the abort flag (used only while unwinding).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > 100000000ull) break;
    }
}

// max(a, b, c) in one instruction (no NaN operands occur here: scores are
// finite or -inf).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Barrier of the softmax threads of one CTA on an mbarrier, so that it shares
// the bounded, abort-aware wait of the pipeline barriers.
__device__ __forceinline__ bool group_sync(uint32_t bar, uint32_t& phase, volatile int* abort,
                                           unsigned* err) {
    mbar_arrive(bar);
    const bool ok = mbar_wait(bar, phase, abort, err);
    phase ^= 1u;
    return ok;
}

// Cluster-scope forms of the barrier operations, for ring slots that the
// converter warps of both CTAs fill with generic stores: the arrive releases
// (and the wait acquires) at cluster scope.
__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait as mbar_wait, with cluster-scope acquire.
__device__ __forceinline__ bool mbar_wait_cl(uint32_t bar, uint32_t parity, volatile int* abort,
                                             unsigned* err) {
    if (mbar_try_wait_cl(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait_cl(bar, parity)) return true;
        if ((n & 63u) == 0) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > kWaitTimeoutNs) {
                *abort = 1;
                atomicOr(err, kErrWaitTimeout);
                return false;
            }
        }
    }
}
// Arrive with cluster-scope release on an mbarrier of this CTA (local) or of
// the pair's even CTA (remote, address from mapa).
__device__ __forceinline__ void arrive_cl_local(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void arrive_cl_remote(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
                 : "memory");
}
// Two E4M3 codes (low 16 bits of v, low byte first) -> fp16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t v) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)v));
    return r;
}
// 16 E4M3 codes -> two 16-byte units of 8 fp16 each.
__device__ __forceinline__ void e4m3x16_f16(const uint4& c, uint4& lo, uint4& hi) {
    lo = make_uint4(e4m3x2_f16x2(c.x), e4m3x2_f16x2(c.x >> 16), e4m3x2_f16x2(c.y),
                    e4m3x2_f16x2(c.y >> 16));
    hi = make_uint4(e4m3x2_f16x2(c.z), e4m3x2_f16x2(c.z >> 16), e4m3x2_f16x2(c.w),
                    e4m3x2_f16x2(c.w >> 16));
}

// MH: the tile space holds one pair-tile range per query head (Hkv > 1,
// 3-D maps); otherwise one range of packed rows (2-D maps).  DH: head size,
// 256 or 128.  F8: K and V are E4M3 codes (read through P.k8 / P.v8; tm_k
// and tm_v are unused), converted to fp16 in shared memory by four extra
// warps.
template <bool MH, int DH, bool F8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg<F8, DH>::NTHREADS, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const Params P) {
    static_assert(DH == 256 || DH == 128, "head size");
    constexpr int SLOTS = DH / 128;                 // ring slots per tile, K and V each
    constexpr int QCH = DH / 64;                    // 64-wide chunks of a Q / K row
    constexpr int QB = BM * DH * 2;                 // this CTA's Q tile bytes
    constexpr int VATOMS = DH / 128;                // 64-wide d atoms of this CTA's V half
    constexpr int SUB_BYTES = 32 * VATOMS * 128;    // one 32-key V sub-tile
    constexpr int SUBS = SLOT_BYTES / SUB_BYTES;    // V sub-tiles per slot
    constexpr int OCOLS = DH / NWG;                 // O columns per softmax thread
    constexpr uint32_t NSB = SBuf<DH>::N;           // S buffers in tensor memory
    // Three S buffers: Q.K^T and P.V come from two threads; two: from one.
    constexpr bool TWO_ISSUERS = NSB == 3;
    constexpr uint32_t IDESC_PV = idesc_f16_f32(256, DH, false, true);
    using C = Cfg<F8, DH>;
    constexpr int NK = C::NK, NRING = C::NRING;
    constexpr int RING_BYTES = C::RING_BYTES, NUM_BARS = C::NUM_BARS;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - smem_u32(smem_raw));
    // Layout: fp16 ring | Q | exchange | barriers | tmem address.
    const uint32_t s_ring = base;
    const uint32_t s_q = base + RING_BYTES;
    const uint32_t s_bars = s_q + Q_BYTES + XCH_BYTES;
    const Bars<NRING> BR{s_bars};
    float* xch = reinterpret_cast<float*>(base_ptr + RING_BYTES + Q_BYTES);
    uint32_t* tmem_base_ptr = reinterpret_cast<uint32_t*>(base_ptr + RING_BYTES + Q_BYTES +
                                                          XCH_BYTES + NUM_BARS * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_ptr + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();      // 0: issues the UMMAs of the pair
    const bool leader = rank == 0;
    const int pair = (int)cluster_id_x();

    if (threadIdx.x == 0) {
        for (int s = 0; s < NRING; ++s) {
            // fp16 path: one arrival (with the pair's transaction bytes); F8: one
            // arrival per converter warp of the role in either CTA.
            mbar_init(BR.full(s), F8 ? 4 : 1);
            mbar_init(BR.empty(s), 1);
        }
        mbar_init(BR.qfull(), 1);
        mbar_init(BR.qempty(), 1);
        for (int i = 0; i < 3; ++i) {
            mbar_init(BR.sfull(i), 1);
            mbar_init(BR.pfull(i), 2 * NSOFT / 32);   // one arrival per softmax warp of the pair
            mbar_init(BR.ofull(i), 1);
        }
        mbar_init(BR.drain(), 1);
        mbar_init(BR.drain2(), 1);
        mbar_init(BR.group(), NSOFT);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    if (warp == 1) {
        // One warp of each CTA of the pair allocates, collectively.
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_base_ptr)),
                     "r"(TMEM_COLS)
                     : "memory");
    }
    tc_fence_before();
    // Both CTAs' barriers are initialised before either uses the other's.
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_ptr;
    // The merge kernel may be scheduled now; it waits for this grid to finish.
    asm volatile("griddepcontrol.launch_dependents;");

    SegIter<MH> it;
    it.init(P, pair);
    int pt, hd, jb, je, n;
    bool is_first;

    if (warp == 0 || warp == V_WARP) {
        // ------------------------------------------------------------ producers
        // Warp 0: Q and K; warp V_WARP: V.  Each loads this CTA's half of
        // every operand; completions land on the even CTA's full barriers,
        // whose transaction count the even CTA sets for both halves.  F8: warp
        // 0 loads Q only (the converter warps fill the K / V slots).
        if (lane == 0 && (!F8 || warp == 0)) {
            const bool kq = warp == 0;
            const int first = kq ? 0 : NK;
            uint32_t t = 0;   // tiles loaded so far (tile t uses S buffer t % NSB)
            int seg = 0;
            bool ok = true;
            while (ok && it.next(P, pt, hd, jb, je, n, is_first)) {
                const int kvh = MH ? hd / P.head_group : 0;   // KV head of this segment
                if (kq) {
                    if (!mbar_wait(BR.qempty(), (seg & 1) ^ 1, abort_flag, P.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t qb = BR.qfull();
                    if (leader) mbar_arrive_expect_tx(qb, 2 * QB);
                    for (int c = 0; c < QCH; ++c)
                        tma_load_pair<MH>(s_q + c * (BM * 128), &tm_q, leader_addr(qb), c * 64, hd,
                                      pt * BM2 + BM * (int)rank);
                }
                for (int j = jb; !F8 && ok && j < je; ++j) {
                    // Tile t's slots are free once the UMMAs of tile t - NSB that
                    // read them have completed: Q.K^T (scores ready) for K, P.V
                    // (O ready) for V, both committed to this CTA's barriers too.
                    const uint32_t u = t % NSB;
                    if (t >= NSB &&
                        !mbar_wait(kq ? BR.sfull(u) : BR.ofull(u), ((t - NSB) / NSB) & 1,
                                   abort_flag, P.err)) {
                        ok = false;
                        break;
                    }
                    const int slot0 = first + (int)u * SLOTS;
                    const uint32_t fb = BR.full(slot0);
                    if (leader) mbar_arrive_expect_tx(fb, 2 * SLOTS * SLOT_BYTES);
                    const uint32_t fbl = leader_addr(fb);
                    for (int h = 0; h < SLOTS; ++h) {
                        const uint32_t dst = s_ring + (slot0 + h) * SLOT_BYTES;
                        if (kq) {
                            // K: d chunks 2h, 2h + 1 of this CTA's 64 keys
                            for (int cc = 0; cc < 2; ++cc)
                                tma_load_pair<MH>(dst + cc * HALF_SLOT, &tm_k, fbl,
                                                  (2 * h + cc) * 64, kvh,
                                                  j * BN + 64 * (int)rank);
                        } else {
                            // V: sub-tiles SUBS h .. SUBS h + SUBS - 1 (32 keys)
                            // x this CTA's DH / 2 d
                            for (int ss = 0; ss < SUBS; ++ss)
                                for (int a = 0; a < VATOMS; ++a)
                                    tma_load_pair<MH>(dst + ss * SUB_BYTES + a * 4096, &tm_v,
                                                      fbl, (DH / 2) * (int)rank + 64 * a, kvh,
                                                      j * BN + (SUBS * h + ss) * 32);
                        }
                    }
                    ++t;
                }
                ++seg;
            }
            if (!ok && leader) {
                // Unwind: let every copy still in flight land before the CTA exits
                // (the even CTA's full barriers count both halves).
                if (!F8) {
                    for (uint32_t u = 0; u < NSB; ++u) {
                        const uint32_t fills = t > u ? (t - u + NSB - 1) / NSB : 0;
                        if (fills) drain_wait(BR.full(first + (int)u * SLOTS), (fills - 1) & 1u);
                    }
                }
                if (kq && seg > 0) drain_wait(BR.qfull(), (seg - 1) & 1);
            }
        }
    } else if (F8 && warp > V_WARP && warp <= V_WARP + C::NCONV) {
        // ------------------------------------------------------------ converters (F8)
        // Warps V_WARP + 1, + 2 convert K, V_WARP + 3, + 4 V, each half of the
        // rows of every slot of a tile.  A lane loads all its 16-byte code
        // chunks of the tile from global memory (L2) first, then waits for the
        // tile's slots to be free (the scores-ready / O-ready barrier of the UMMAs
        // NSB tiles back, as the fp16 copies do), writes the fp16 values exactly
        // where the fp16 path's TMA would have put them (128-byte-swizzled rows),
        // makes them visible to the tensor cores' async proxy and arrives
        // (cluster scope) on the even CTA's full barrier.  E4M3 -> fp16 is
        // exact; keys past KV are zero codes, as the TMA's fill would be.
        const int cw = warp - V_WARP - 1;           // 0..3
        const bool kc = cw < 2;
        const int part = cw & 1;                    // which half of the slot's rows
        // Slot rows: K 64 keys x 128 codes; V (BN / SLOTS) keys x DH / 2 codes.
        constexpr int RBV = DH / 2;                 // V code bytes per row
        constexpr int RPIK = 32 / (128 / 16);       // K rows per warp pass (4)
        constexpr int RPIV = 32 / (RBV / 16);       // V rows per warp pass (4 or 8)
        constexpr int PASSES = 8;                   // passes per warp per slot (half a slot)
        static_assert(64 / 2 == RPIK * PASSES && (BN / SLOTS) / 2 == RPIV * PASSES, "passes");
        const int rb = kc ? 128 : RBV;
        const int cpr = rb / 16;                    // 16-code chunks per row
        const int rpi = kc ? RPIK : RPIV;
        const int rbase = part * rpi * PASSES + lane / cpr;
        const int c = lane % cpr;                   // 16 codes: d 16c .. 16c + 15 of the row
        const uint8_t* codes = kc ? P.k8 : P.v8;
        const int first = kc ? 0 : NK;
        uint32_t t = 0;
        bool ok = true;
        while (ok && it.next(P, pt, hd, jb, je, n, is_first)) {
            const int kvh = MH ? hd / P.head_group : 0;
            for (int j = jb; ok && j < je; ++j) {
                uint4 code[SLOTS][PASSES];
#pragma unroll
                for (int h = 0; h < SLOTS; ++h) {
                    // K slot h: this CTA's keys j BN + 64 rank + r, d 128 h ..; V slot h:
                    // keys j BN + h (BN / SLOTS) + r, this CTA's d (DH / 2) rank ..
                    const int key0 = kc ? j * BN + 64 * (int)rank : j * BN + h * (BN / SLOTS);
                    const int d0 = (kc ? 128 * h : (DH / 2) * (int)rank) + 16 * c;
#pragma unroll
                    for (int i = 0; i < PASSES; ++i) {
                        const int key = key0 + rbase + i * rpi;
                        code[h][i] = key < P.KV
                                         ? __ldg(reinterpret_cast<const uint4*>(
                                               codes + (size_t)key * P.kv_rs + kvh * DH + d0))
                                         : make_uint4(0, 0, 0, 0);
                    }
                }
                const uint32_t u = t % NSB;
                if (t >= NSB)
                    ok = mbar_wait(kc ? BR.sfull(u) : BR.ofull(u), ((t - NSB) / NSB) & 1,
                                   abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                const int slot0 = first + (int)u * SLOTS;
#pragma unroll
                for (int h = 0; h < SLOTS; ++h) {
                    uint8_t* dst = base_ptr + (slot0 + h) * SLOT_BYTES;
#pragma unroll
                    for (int i = 0; i < PASSES; ++i) {
                        const int r = rbase + i * rpi;
                        uint4 lo, hi;
                        e4m3x16_f16(code[h][i], lo, hi);
                        // K slot: chunk c / 4 (64 d) of HALF_SLOT, row r; V slot:
                        // sub-tile r / 32, atom c / 4 (64 d), row r % 32.
                        const uint32_t o =
                            kc ? (uint32_t)((c >> 2) * HALF_SLOT + r * 128)
                               : (uint32_t)((r >> 5) * SUB_BYTES + (c >> 2) * 4096 + (r & 31) * 128);
                        const uint32_t u0 = 2u * (uint32_t)(c & 3), sw = (uint32_t)(r & 7);
                        *reinterpret_cast<uint4*>(dst + o + ((u0 ^ sw) << 4)) = lo;
                        *reinterpret_cast<uint4*>(dst + o + (((u0 + 1) ^ sw) << 4)) = hi;
                    }
                }
                // Order the generic stores before the tensor cores' reads of this
                // CTA's shared memory (reached through the cluster window by the
                // even CTA's UMMAs); a shared-memory-only proxy fence.
                asm volatile("fence.proxy.async.shared::cluster;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    if (leader) arrive_cl_local(BR.full(slot0));
                    else arrive_cl_remote(leader_addr(BR.full(slot0)));
                }
                ++t;
            }
        }
    } else if (warp == 1 || warp == C::PV_WARP) {
      if (lane == 0 && leader && (TWO_ISSUERS || warp == 1)) {
        // ------------------------------------------------------------ UMMA issuers
        // Each UMMA issues at about the tensor pipe's own rate, so the issuing
        // thread's barrier waits and commits (several hundred cycles per tile)
        // leave the pipe idle unless something else issues meanwhile.  With
        // three S buffers (DH = 128) two threads of the even CTA issue: warp 1
        // every Q.K^T, warp PV_WARP every P.V, and Q.K^T of tile g waits only
        // for the P.V of tile g - 3 (its buffer's O-ready barrier), so the chain
        // softmax -> P.V -> Q.K^T spans three tiles.  With two (DH = 256, where O takes half of
        // tensor memory) warp 1 issues both in one stream: Q.K^T of tile g + 1,
        // then P.V of tile g, the tensor pipe's order keeping Q.K^T of tile
        // g + 2 behind the P.V of tile g that reads the same buffer.
        const bool qk_role = warp == 1;
        uint32_t g = 0;
        int seg = 0;
        bool ok = true;
        // Tile gg's K (V) slots are first + (gg % NSB) * SLOTS .., landed when
        // the first one's full barrier completes phase gg / NSB.  A TMA copy and
        // the UMMA that reads it are both async-proxy operations ordered by the
        // mbarrier's completion, so no tcgen05 fence is needed; F8: the slots
        // were filled by generic stores of both CTAs' converter warps, which
        // arrive with cluster-scope release, so acquire at cluster scope.
        auto take_tile = [&](int first, uint32_t gg, int& slot0) -> bool {
            slot0 = first + (int)(gg % NSB) * SLOTS;
            if constexpr (F8) return mbar_wait_cl(BR.full(slot0), (gg / NSB) & 1, abort_flag, P.err);
            return mbar_wait(BR.full(slot0), (gg / NSB) & 1, abort_flag, P.err);
        };
        auto s_col_of = [&](uint32_t gg) { return SBuf<DH>::COL0 + (gg % NSB) * BN; };
        // Descriptor low words: Q chunk c at q_lo + c * (BM * 128 >> 4); a K
        // slot's chunk cc at + cc * (HALF_SLOT >> 4); a K step of 16
        // elements (32 bytes) at + 2.
        const uint32_t q_lo = desc_lo(s_q, 16);
        auto issue_qk = [&](uint32_t gg) -> bool {
            const uint32_t d = tmem + s_col_of(gg);
            int slot0 = 0;
            if (!take_tile(0, gg, slot0)) return false;
#pragma unroll
            for (int h = 0; h < SLOTS; ++h) {
                const int slot = slot0 + h;
                const uint32_t k_lo = desc_lo(s_ring + slot * SLOT_BYTES, 16);
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int c = 2 * h + cc;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t a = desc64(q_lo + c * ((BM * 128) >> 4) + kk * 2);
                        const uint64_t b = desc64(k_lo + cc * (HALF_SLOT >> 4) + kk * 2);
                        if (c == 0 && kk == 0)
                            umma_ss_pair_c<false>(d, a, b, IDESC_QK);
                        else
                            umma_ss_pair_c<true>(d, a, b, IDESC_QK);
                    }
                }
            }
            return true;
        };
        auto issue_pv = [&](uint32_t gg, bool acc0) -> bool {
            const uint32_t p_base = tmem + s_col_of(gg);
            int slot0 = 0;
            if (!take_tile(NK, gg, slot0)) return false;
#pragma unroll
            for (int h = 0; h < SLOTS; ++h) {
                const int slot = slot0 + h;
                // V: MN-major, 64-element atoms 4096 B apart (LBO), 8-key groups
                // 1024 B apart (SBO); a K step of 16 keys is 2048 B.
                const uint32_t v_lo = desc_lo(s_ring + slot * SLOT_BYTES, 4096);
#pragma unroll
                for (int ss = 0; ss < SUBS; ++ss) {
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        const uint64_t b = desc64(v_lo + ss * (SUB_BYTES >> 4) + ks * (2048 >> 4));
                        // P of keys kb .. kb + 15: part kb / COLS sits at columns
                        // COLS (kb / COLS) + (kb % COLS) / 2 of the S buffer.
                        const int kb = (SUBS * h + ss) * 32 + ks * 16;
                        const uint32_t a_tmem = p_base + (kb / COLS) * COLS + (kb % COLS) / 2;
                        if (h == 0 && ss == 0 && ks == 0)
                            umma_ts_pair(tmem + O_COL, a_tmem, b, IDESC_PV, acc0 ? 1u : 0u);
                        else
                            umma_ts_pair_c<true>(tmem + O_COL, a_tmem, b, IDESC_PV);
                    }
                }
            }
            return true;
        };
        while (ok && it.next(P, pt, hd, jb, je, n, is_first)) {
            if (qk_role) {
                if (!mbar_wait(BR.qfull(), seg & 1, abort_flag, P.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            if (TWO_ISSUERS) {
                for (int j = jb; ok && j < je; ++j) {
                    const uint32_t gg = g + (j - jb);
                    if (qk_role) {
                        // S buffer gg % NSB is free once the P.V of tile gg - NSB
                        // (which read its P) has completed.
                        if (gg >= NSB) {
                            ok = mbar_wait(BR.ofull(gg % NSB), ((gg - NSB) / NSB) & 1, abort_flag,
                                           P.err);
                            if (!ok) break;
                            tc_fence_after();
                        }
                        ok = issue_qk(gg);
                        if (!ok) break;
                        umma_commit_pair(BR.sfull(gg % NSB));
                        if (j == je - 1) umma_commit_pair(BR.qempty());
                    } else {
                        ok = mbar_wait(BR.pfull(gg % NSB), (gg / NSB) & 1, abort_flag, P.err);
                        if (!ok) break;
                        tc_fence_after();
                        ok = issue_pv(gg, j > jb);
                        if (!ok) break;
                        umma_commit_pair(BR.ofull(gg % NSB));
                    }
                }
            } else {
                ok = issue_qk(g);
                if (!ok) break;
                umma_commit_pair(BR.sfull(g & 1));
                if (je - jb == 1) umma_commit_pair(BR.qempty());
                for (int j = jb; j < je; ++j) {
                    const uint32_t gg = g + (j - jb);
                    if (j + 1 < je) {
                        ok = issue_qk(gg + 1);
                        if (!ok) break;
                        umma_commit_pair(BR.sfull((gg + 1) & 1));
                        if (j + 1 == je - 1) umma_commit_pair(BR.qempty());
                    }
                    if (!mbar_wait(BR.pfull(gg & 1), (gg >> 1) & 1, abort_flag, P.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    ok = issue_pv(gg, j > jb);
                    if (!ok) break;
                    umma_commit_pair(BR.ofull(gg & 1));
                }
            }
            g += je - jb;
            ++seg;
        }
        if (!ok) {
            // Unwind: wait for every UMMA this thread issued before TMEM is freed.
            const uint32_t db = qk_role ? BR.drain() : BR.drain2();
            umma_commit_pair(db);
            drain_wait(db, 0);
        }
      }
    } else if (warp < V_WARP) {
        // ------------------------------------------------------------ softmax / epilogue
        // Warpgroup hg owns S columns [COLS hg, COLS (hg + 1)) of every tile
        // and O columns [OCOLS hg, OCOLS (hg + 1)).  Row maxima: each thread
        // writes its part maximum to xch[tile parity][hg][row]; after the group
        // barrier it reads the others', so all threads of a row see the same
        // maximum (combined in a fixed order).
        const int hg = (warp - 2) >> 2;
        const int wq = warp & 3;           // TMEM lane quarter this warp may access
        const int row = wq * 32 + lane;    // tile row == TMEM lane
        const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
        float* xl = xch + 2 * NWG * BM;    // row-sum parts [hg][row]
        const uint32_t gbar = BR.group();
        uint32_t gphase = 0;
        // F8: the K scale joins the score scale; the V scale multiplies O.
        const float sl2 = F8 ? P.scale_log2 * __ldg(P.kscale) : P.scale_log2;
        const float vsc = F8 ? __ldg(P.vscale) : 1.0f;
        uint32_t g = 0;
        bool ok = true;
        while (ok && it.next(P, pt, hd, jb, je, n, is_first)) {
            const int m_row = pt * BM2 + BM * (int)rank + row;
            const bool valid = m_row < P.M_total;
            const int lim = P.KV - P.Q + P.grp.div(m_row);      // last visible key
            const int j_mask = (P.KV - P.Q + P.grp.div(pt * BM2 + BM * (int)rank) + 1) / BN;
            float m_ref = -INFINITY;
            float l = 0.f;
            for (int j = jb; j < je; ++j) {
                const uint32_t gg = g + (j - jb);
                const uint32_t sb = gg % NSB;
                const uint32_t s_col = SBuf<DH>::COL0 + sb * BN;
                ok = mbar_wait(BR.sfull(sb), (gg / NSB) & 1, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                uint32_t sr[COLS];
#pragma unroll
                for (int c = 0; c < COLS / 32; ++c)
                    tmem_ld32(t_lane + s_col + COLS * hg + 32 * c,
                              *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
                tmem_ld_wait<COLS>(sr);
                float* s = reinterpret_cast<float*>(sr);
                if (j >= j_mask) {
                    const int k0 = j * BN + COLS * hg;
#pragma unroll
                    for (int c = 0; c < COLS; ++c)
                        if (k0 + c > lim) s[c] = -INFINITY;
                }
                // Four independent chains (columns i, i + 4, ..., i + COLS - 4) of
                // three-input maxima, two columns per instruction.
                static_assert(COLS % 8 == 0, "row max chains");
                float cm[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float m = fmax3(s[i], s[i + 4], s[i + 8]);
#pragma unroll
                    for (int k = 3; k + 1 < COLS / 4; k += 2)
                        m = fmax3(m, s[i + 4 * k], s[i + 4 * k + 4]);
                    cm[i] = fmaxf(m, s[i + COLS - 4]);
                }
                const float hm = fmax3(cm[0], cm[1], fmaxf(cm[2], cm[3]));
                float* xp = xch + (gg & 1) * (NWG * BM);
                xp[hg * BM + row] = hm;
                ok = group_sync(gbar, gphase, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                float rm = xp[row];
#pragma unroll
                for (int h = 1; h < NWG; ++h) rm = fmaxf(rm, xp[h * BM + row]);
                const float mx = rm * sl2;
                if (j == jb) {
                    m_ref = mx;
                } else {
                    const bool need = mx > m_ref + RESCALE_THRESHOLD;
                    if (__any_sync(0xffffffffu, need)) {
                        ok = mbar_wait(BR.ofull((gg - 1) % NSB), ((gg - 1) / NSB) & 1,
                                       abort_flag, P.err);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                        tc_fence_after();
                        const float f = need ? ex2(m_ref - mx) : 1.0f;
                        if (need) {
                            l *= f;
                            m_ref = mx;
                        }
#pragma unroll 1
                        for (int c = 0; c < OCOLS / 32; ++c) {
                            uint32_t o[32];
                            const uint32_t oc = O_COL + OCOLS * hg + 32 * c;
                            tmem_ld32(t_lane + oc, o);
                            tmem_ld_wait<32>(o);
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                            tmem_st32(t_lane + oc, o);
                        }
                        tmem_st_wait();
                    }
                }
                const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
                float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
                uint32_t pk[COLS / 2];
#pragma unroll
                for (int e = 0; e < COLS / 2; e += 2) {
                    const int c = 2 * e;
                    const float p0 = ex2(fmaf(s[c], sl2, neg));
                    const float p1 = ex2(fmaf(s[c + 1], sl2, neg));
                    const float p2 = ex2(fmaf(s[c + 2], sl2, neg));
                    const float p3 = ex2(fmaf(s[c + 3], sl2, neg));
                    l0 += p0;
                    l1 += p1;
                    l2 += p2;
                    l3 += p3;
                    pk[e] = pack_half2(p0, p1);
                    pk[e + 1] = pack_half2(p2, p3);
                }
                tmem_st32(t_lane + s_col + COLS * hg, pk);
                l += (l0 + l1) + (l2 + l3);
                tmem_st_wait();
                // No wait for the previous tile's P.V here unless O was rescaled
                // above: P(j) goes into S buffer j % NSB, whose last reader (the
                // P.V of tile j - NSB) had completed before the Q.K^T of tile j
                // was issued, and the O-ready barriers cannot run more than one
                // phase ahead of this thread (their next phase needs its P).
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (leader) mbar_arrive(BR.pfull(sb));
                    else remote_arrive(leader_addr(BR.pfull(sb)));
                }
            }
            if (!ok) break;
            // ---------------------------------------------------------- epilogue
            const uint32_t gl = g + (je - jb) - 1;
            ok = mbar_wait(BR.ofull(gl % NSB), (gl / NSB) & 1, abort_flag, P.err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            // Row sum: the parts, added in a fixed order.
            xl[hg * BM + row] = l;
            ok = group_sync(gbar, gphase, abort_flag, P.err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            float l_row = xl[row];
#pragma unroll
            for (int h = 1; h < NWG; ++h) l_row += xl[h * BM + row];
            if (jb == 0 && je == n) {
                const float inv = (l_row > 0.f) ? vsc / l_row : 0.f;
                uint4* dst = reinterpret_cast<uint4*>(P.out + (MH ? (size_t)hd * DH : 0) + (size_t)m_row * P.out_stride + OCOLS * hg);
#pragma unroll 1
                for (int c = 0; c < OCOLS / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(t_lane + O_COL + OCOLS * hg + 32 * c, o);
                    tmem_ld_wait<32>(o);
                    uint32_t hv[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        hv[e] = pack_half2(__uint_as_float(o[2 * e]) * inv,
                                           __uint_as_float(o[2 * e + 1]) * inv);
                    if (valid) {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[c * 4 + e] = make_uint4(hv[4 * e], hv[4 * e + 1], hv[4 * e + 2],
                                                        hv[4 * e + 3]);
                    }
                }
            } else {
                const int slot = is_first ? 0 : 1;
                const size_t prow = ((size_t)pair * 2 + slot) * BM2 + BM * rank + row;
                uint4* dst = reinterpret_cast<uint4*>(P.ws_o + prow * DH + OCOLS * hg);
#pragma unroll 1
                for (int c = 0; c < OCOLS / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(t_lane + O_COL + OCOLS * hg + 32 * c, o);
                    tmem_ld_wait<32>(o);
                    if (F8) {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            o[e] = __float_as_uint(__uint_as_float(o[e]) * vsc);
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dst[c * 8 + e] = make_uint4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
                }
                if (hg == 0) {
                    P.ws_ml[prow * 2 + 0] = m_ref;
                    P.ws_ml[prow * 2 + 1] = l_row;
                }
            }
            g += je - jb;
        }
    }

    // After an abort, give copies the other CTA of the pair still had in
    // flight into this CTA's shared memory time to land before it exits.
    __syncthreads();
    if (*abort_flag) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 1000000ull) {
        }
    }
    tc_fence_before();
    // Neither CTA leaves while the other may still signal its barriers.
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

// A pair tile cut between pairs c0 .. c_last: its first piece is pair c0's
// last segment (partial slot slot0), the others are the first segments (slot
// 0) of pairs c0 + 1 .. c_last.  Found on the host from the same shape-only
// schedule.
struct MergeTasks {
    int n;
    int4 task[kMaxClusters];  // (tile-space index, c0, slot0, c_last)
};

// blockIdx.x picks a cut pair tile, blockIdx.y 8 of its 256 rows; thread
// (row, lane) merges 8 consecutive d (lanes past DH / 8 have none).  Pieces
// are combined in pair order
// (exact log-sum-exp merge), so the result does not depend on timing.  The
// kernel is a programmatic dependent of the main kernel: its launch overlaps
// that kernel's tail, and griddepcontrol.wait holds it until the partials are
// complete.
template <bool MH, int DH>
__global__ void __launch_bounds__(256)
prefill_merge_kernel(const Params P, const __grid_constant__ MergeTasks T) {
    const int4 tk = T.task[blockIdx.x];
    const int t = tk.x, c0 = tk.y, slot0 = tk.z, c_last = tk.w;
    const int hd = MH ? P.ptiles.div(t) : 0;        // head of tile-space index t
    const int r = blockIdx.y * 8 + (threadIdx.x >> 5);
    const int m_row = (t - hd * P.num_ptiles) * BM2 + r;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (m_row >= P.M_total) return;
    const int d0 = (threadIdx.x & 31) * 8;
    if (d0 >= DH) return;
    float M = -INFINITY;
    for (int c = c0; c <= c_last; ++c) {
        const size_t prow = ((size_t)c * 2 + (c == c0 ? slot0 : 0)) * BM2 + r;
        M = fmaxf(M, P.ws_ml[prow * 2]);
    }
    float L = 0.f;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int c = c0; c <= c_last; ++c) {
        const size_t prow = ((size_t)c * 2 + (c == c0 ? slot0 : 0)) * BM2 + r;
        const float mp = P.ws_ml[prow * 2];
        const float w = (mp == -INFINITY) ? 0.f : exp2f(mp - M);
        L += P.ws_ml[prow * 2 + 1] * w;
        const float4* o = reinterpret_cast<const float4*>(P.ws_o + prow * DH + d0);
        const float4 a = o[0], b = o[1];
        acc[0] += a.x * w; acc[1] += a.y * w; acc[2] += a.z * w; acc[3] += a.w * w;
        acc[4] += b.x * w; acc[5] += b.y * w; acc[6] += b.z * w; acc[7] += b.w * w;
    }
    const float inv = L > 0.f ? 1.0f / L : 0.f;
    uint4 hv = make_uint4(pack_half2(acc[0] * inv, acc[1] * inv), pack_half2(acc[2] * inv, acc[3] * inv),
                          pack_half2(acc[4] * inv, acc[5] * inv), pack_half2(acc[6] * inv, acc[7] * inv));
    *reinterpret_cast<uint4*>(P.out + (MH ? (size_t)hd * DH : 0) + (size_t)m_row * P.out_stride + d0) = hv;
}

// Host side of the schedule: the cut pair tiles and their pieces.
static void find_cut_tiles(const Params& P, MergeTasks& T) {
    T.n = 0;
    long long cum = 0;
    int c = 0;  // first pair whose range ends after cum
    for (int t = 0; t < P.heads * P.num_ptiles; ++t) {
        const int n = kv_tiles(t % P.num_ptiles, P.Q, P.KV, P.M_total, P.grp);
        const long long t_end = cum + n;
        // pair holding the tile's first iteration
        while (c + 1 < P.G && pair_begin(P.total, P.G, c + 1) <= cum) ++c;
        if (pair_begin(P.total, P.G, c + 1) < t_end) {  // the tile continues past pair c
            int c_last = c + 1;
            while (c_last + 1 < P.G && pair_begin(P.total, P.G, c_last + 1) < t_end) ++c_last;
            const int slot0 = (pair_begin(P.total, P.G, c) == cum) ? 0 : 1;
            T.task[T.n++] = make_int4(t, c, slot0, c_last);
        }
        cum = t_end;
    }
}

// Pairs that can be resident at once with this kernel's shared memory (the
// SMs of a pair must share a GPC, so this can be below num_sms / 2).
static int max_pairs(int device) {
    static std::atomic<int> cached[64];   // 0 until known (static storage starts at 0)
    if (device < 64) {
        const int c = cached[device].load(std::memory_order_relaxed);
        if (c) return c;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(Cfg<false, 256>::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg<false, 256>::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    // All instantiations use one CTA per SM (their shared memory allows no
    // second), so the fp16 kernel's count holds for all.
    if (cudaOccupancyMaxActiveClusters(&n, prefill_kernel<false, 256, false>, &cfg) != cudaSuccess ||
        n < 1) {
        cudaGetLastError();
        return 0;
    }
    if (n > kMaxClusters) n = kMaxClusters;
    if (device < 64) cached[device].store(n, std::memory_order_relaxed);
    return n;
}

// One main-kernel launch and, when pair tiles were cut, its merge.
template <bool MH, int DH, bool F8>
static int launch_one(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const Params& P, const MergeTasks& tasks, cudaStream_t stream) {
    using C = Cfg<F8, DH>;
    if (ensure_smem_limit(reinterpret_cast<const void*>(prefill_kernel<MH, DH, F8>),
                          C::SMEM_BYTES) != GQA_OK)
        return GQA_ERR_CUDA;
    prefill_kernel<MH, DH, F8><<<2 * P.G, C::NTHREADS, C::SMEM_BYTES, stream>>>(tq, tk, tv, P);
    if (cudaGetLastError() != cudaSuccess) return GQA_ERR_CUDA;
    if (tasks.n > 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(tasks.n, BM2 / 8);
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, prefill_merge_kernel<MH, DH>, P, tasks) != cudaSuccess)
            return GQA_ERR_CUDA;
    }
    return GQA_OK;
}

}  // namespace prefill

int prefill_resident_pairs() {
    const DeviceInfo* di = device_info();
    if (!di) return -1;
    if (ensure_smem_limit(reinterpret_cast<const void*>(prefill::prefill_kernel<false, 256, false>),
                          prefill::Cfg<false, 256>::SMEM_BYTES) != GQA_OK)
        return -1;
    return prefill::max_pairs(di->device);
}

size_t prefill_workspace_bytes(int Q, int KV, int num_sms) {
    (void)Q;
    (void)KV;
    const size_t per_pair = (size_t)2 * prefill::BM2 * (prefill::D + 2) * sizeof(float);
    const size_t pairs = (size_t)(num_sms / 2 > 0 ? num_sms / 2 : 1);
    return kWorkspaceCounterBytes + per_pair * pairs + 256;
}

int prefill_launch(const void* q, const void* k, const void* v, const float* kscale,
                   const float* vscale, void* out, int Q, int KV, int Hq, int Hkv, int Dh,
                   float scale, cudaStream_t stream) {
    using namespace prefill;
    const DeviceInfo* di = device_info();
    if (!di) return GQA_ERR_CUDA;
    const bool f8 = kscale != nullptr;   // K / V are E4M3 codes with device-side scales
    if (ensure_smem_limit(reinterpret_cast<const void*>(prefill_kernel<false, 256, false>),
                          Cfg<false, 256>::SMEM_BYTES) != GQA_OK)
        return GQA_ERR_CUDA;
    const int pairs_max = max_pairs(di->device);
    if (pairs_max < 1) return GQA_ERR_CUDA;
    // Query heads that share the single KV head are packed (positions x Hq
    // rows of one head of the tile space); with several KV heads every query
    // head is a head of the tile space, with one row per position, in the
    // same launch.  The tensor maps are (d, head, row) either way.
    const bool packed = (Hkv == 1);
    const int grp = packed ? Hq : 1;
    Params P;
    P.Q = Q;
    P.KV = KV;
    P.heads = packed ? 1 : Hq;
    P.head_group = packed ? 1 : Hq / Hkv;
    P.grp = make_fastdiv(grp);
    P.out_stride = packed ? Dh : Hq * Dh;
    P.M_total = Q * grp;
    P.num_ptiles = (P.M_total + BM2 - 1) / BM2;
    P.ptiles = make_fastdiv(P.num_ptiles);
    long long total = 0;
    for (int t = 0; t < P.num_ptiles; ++t) total += kv_tiles(t, Q, KV, P.M_total, P.grp);
    total *= P.heads;
    P.total = total;
    int G = pairs_max < di->num_sms / 2 ? pairs_max : di->num_sms / 2;
    if (G < 1) G = 1;
    P.G = (int)(total < G ? total : G);
    P.scale_log2 = scale * 1.4426950408889634f;
    P.kscale = kscale;
    P.vscale = vscale;
    P.k8 = f8 ? static_cast<const uint8_t*>(k) : nullptr;
    P.v8 = f8 ? static_cast<const uint8_t*>(v) : nullptr;
    P.kv_rs = Hkv * Dh;
    P.err = di->err_word;
    P.out = static_cast<__half*>(out);

    void* ws;
    size_t ws_bytes;
    current_workspace(&ws, &ws_bytes);
    const size_t need = kWorkspaceCounterBytes + (size_t)P.G * 2 * BM2 * (D + 2) * sizeof(float);
    if (P.G > 1 && (!ws || ws_bytes < need)) return GQA_ERR_WORKSPACE;
    if (ws) {
        float* w = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kWorkspaceCounterBytes);
        P.ws_o = w;
        P.ws_ml = w + (size_t)P.G * 2 * BM2 * D;
    } else {
        P.ws_o = nullptr;
        P.ws_ml = nullptr;
    }
    MergeTasks tasks;  // passed to the merge kernel by value
    find_cut_tiles(P, tasks);

    // E4M3 K / V are read by the converter warps through P.k8 / P.v8; their
    // kernels take the Q map in the K / V map arguments, unused.
    CUtensorMap tq, tk, tv;
    if (packed) {
        if (!make_map_2d_f16(&tq, q, (uint64_t)P.M_total, Dh, Dh, BM, 64)) return GQA_ERR_CUDA;
        if (f8)
            return Dh == 256 ? launch_one<false, 256, true>(tq, tq, tq, P, tasks, stream)
                             : launch_one<false, 128, true>(tq, tq, tq, P, tasks, stream);
        if (!make_map_2d_f16(&tk, k, (uint64_t)KV, Dh, Dh, BN / 2, 64) ||
            !make_map_2d_f16(&tv, v, (uint64_t)KV, Dh, Dh, 32, 64))
            return GQA_ERR_CUDA;
        return Dh == 256 ? launch_one<false, 256, false>(tq, tk, tv, P, tasks, stream)
                         : launch_one<false, 128, false>(tq, tk, tv, P, tasks, stream);
    }
    const uint64_t row_bytes = 2ull * Dh;
    if (!make_map_3d_f16(&tq, q, Dh, (uint64_t)Hq, (uint64_t)Q, row_bytes,
                         (uint64_t)Hq * row_bytes, BM))
        return GQA_ERR_CUDA;
    if (f8)
        return Dh == 256 ? launch_one<true, 256, true>(tq, tq, tq, P, tasks, stream)
                         : launch_one<true, 128, true>(tq, tq, tq, P, tasks, stream);
    if (!make_map_3d_f16(&tk, k, Dh, (uint64_t)Hkv, (uint64_t)KV, row_bytes,
                         (uint64_t)Hkv * row_bytes, BN / 2) ||
        !make_map_3d_f16(&tv, v, Dh, (uint64_t)Hkv, (uint64_t)KV, row_bytes,
                         (uint64_t)Hkv * row_bytes, 32))
        return GQA_ERR_CUDA;
    return Dh == 256 ? launch_one<true, 256, false>(tq, tk, tv, P, tasks, stream)
                     : launch_one<true, 128, false>(tq, tk, tv, P, tasks, stream);
}

}  // namespace gqa
