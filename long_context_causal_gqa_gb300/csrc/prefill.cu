// prefill.cu -- dense causal GQA prefill on sm_103a.
//
// Problem ("[Kernel][SM70] Default long-prefill GQA architecture", Purpose):
// q [Q, 6, 256], k/v [KV, 1, 256] fp16, scale 1/16, query row i bottom-right
// aligned (sees keys 0 .. KV - Q + i), fp16 output.  The page packs the six
// query heads that share the KV head into wide QK / PV GEMMs and merges the
// causal tail with online-softmax state; both ideas carry over, re-shaped for
// tcgen05:
//
// * Head packing.  q is [Q, 6, 256] = [6Q, 256] row-major, so 128 consecutive
//   flattened rows (about 21 positions x 6 heads) are one 128-row M tile with
//   no padding.  Each K/V tile is read once per 128 packed rows.
// * One CTA per SM, warp-specialised:
//     warp 0      TMA producer (Q tile, then a ring of 16 KB K / V chunks)
//     warp 1      tensor-memory allocation and the single UMMA-issuing thread
//     warps 2..9  softmax + epilogue: two warpgroups, each thread one tile row
//                 (TMEM lane) and half of its columns
// * Tensor memory (512 columns x 128 lanes): O = 256 fp32 columns; two S
//   buffers of 128 fp32 columns, so Q.K^T of tile j+1 runs while tile j's
//   softmax runs.  Each warpgroup's P (fp16) overwrites the first 32 columns
//   of its own 64-column half of the S buffer and feeds P.V straight from
//   tensor memory.  The two threads of a row swap their half maxima through
//   shared memory each tile, so both take the same rescale decisions.
// * Online softmax with a lazy rescale: the per-row reference max only moves
//   (and O is rescaled in TMEM) when a tile's max exceeds it by more than
//   8 (log2 units), which bounds P by 256.
// * Only the one or two KV tiles on a q-tile's diagonal are masked.
// * Work split: the causal-visible (q-tile, kv-tile) iterations are laid out
//   q-tile-major and cut into one contiguous, equal range per CTA (shape-only,
//   so deterministic).  A q-tile cut between CTAs leaves (O, m, l) partials in
//   the workspace; a merge kernel combines them in CTA order (exact
//   log-sum-exp merge).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"
#include "sm100.cuh"

namespace gqa {
namespace prefill {

constexpr int BM = 128;         // packed query rows per tile
constexpr int BN = 128;         // keys per KV tile
constexpr int D = kHeadDim;     // 256
constexpr int HQ = kHq;         // 6
constexpr int NSLOT = 9;        // ring slots
constexpr int SLOT_BYTES = 16384;
constexpr int Q_BYTES = BM * D * 2;           // 64 KB
constexpr int RING_BYTES = NSLOT * SLOT_BYTES;
constexpr int NUM_BARS = 2 * NSLOT + 9;  // full/empty ring, q, s[2], p[2], o, drain, group
constexpr int XCH_BYTES = (2 * 2 + 2) * BM * 4;  // half maxima [parity][half][row], sums [half][row]
constexpr int SMEM_BYTES =
    1024 /*align slack*/ + RING_BYTES + Q_BYTES + XCH_BYTES + NUM_BARS * 8 + 16;
constexpr int NTHREADS = 320;
constexpr int NSOFT = 256;      // softmax threads
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t O_COL = 0;
constexpr uint32_t S_COL0 = 256;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units

// UMMA shapes: S[128 x 128] = Q[128 x 16] K^T, both K-major;
// O[128 x 256] += P[128 x 16] (tensor memory) V[16 x 256], V MN-major.
constexpr uint32_t IDESC_QK = idesc_f16_f32(128, 128, false, false);
constexpr uint32_t IDESC_PV = idesc_f16_f32(128, 256, false, true);

struct Params {
    int Q, KV, M_total, num_qtiles, G;
    long long total;      // causal-visible (q-tile, kv-tile) iterations
    float scale_log2;     // scale * log2(e)
    __half* out;
    float* ws_o;          // [G][2][BM][D] unnormalised partial O
    float* ws_ml;         // [G][2][BM][2] partial (m in log2 units, l)
    unsigned* err;
};

// KV tiles q-tile t needs: up to the last visible key of its last valid row.
__host__ __device__ inline int kv_tiles(int t, int Q, int KV, int M_total) {
    int last = min(t * BM + BM - 1, M_total - 1);
    return (KV - Q + last / HQ) / BN + 1;
}

__host__ __device__ inline long long cta_begin(long long total, int G, int c) {
    return (long long)c * total / G;
}

// Walks the segments (q-tile, [jb, je)) of one CTA's iteration range.
struct SegIter {
    long long pos, end, cum;
    int t;
    bool first;
    __device__ void init(const Params& P, int cta) {
        pos = cta_begin(P.total, P.G, cta);
        end = cta_begin(P.total, P.G, cta + 1);
        t = 0;
        cum = 0;
        first = true;
        while (t < P.num_qtiles) {
            int n = kv_tiles(t, P.Q, P.KV, P.M_total);
            if (cum + n > pos) break;
            cum += n;
            ++t;
        }
    }
    // Next segment; is_first tells whether it is this CTA's first segment.
    __device__ bool next(const Params& P, int& qt, int& jb, int& je, int& n, bool& is_first) {
        if (pos >= end) return false;
        n = kv_tiles(t, P.Q, P.KV, P.M_total);
        qt = t;
        jb = (int)(pos - cum);
        long long e = end - cum;
        je = e < n ? (int)e : n;
        is_first = first;
        first = false;
        pos = cum + je;
        if (je == n) {
            cum += n;
            ++t;
        }
        return true;
    }
};


__device__ __forceinline__ uint32_t bar_full(uint32_t b, int s) { return b + 8 * s; }
__device__ __forceinline__ uint32_t bar_empty(uint32_t b, int s) { return b + 8 * (NSLOT + s); }
__device__ __forceinline__ uint32_t bar_qfull(uint32_t b) { return b + 8 * (2 * NSLOT); }
__device__ __forceinline__ uint32_t bar_qempty(uint32_t b) { return b + 8 * (2 * NSLOT + 1); }
__device__ __forceinline__ uint32_t bar_sfull(uint32_t b, int i) {
    return b + 8 * (2 * NSLOT + 2 + i);
}
__device__ __forceinline__ uint32_t bar_pfull(uint32_t b, int i) {
    return b + 8 * (2 * NSLOT + 4 + i);
}
__device__ __forceinline__ uint32_t bar_ofull(uint32_t b) { return b + 8 * (2 * NSLOT + 6); }
__device__ __forceinline__ uint32_t bar_drain(uint32_t b) { return b + 8 * (2 * NSLOT + 7); }
__device__ __forceinline__ uint32_t bar_group(uint32_t b) { return b + 8 * (2 * NSLOT + 8); }

// Barrier of the 256 softmax threads on an mbarrier, so that it shares the
// bounded, abort-aware wait of the pipeline barriers.
__device__ __forceinline__ bool group_sync(uint32_t bar, uint32_t& phase, volatile int* abort,
                                           unsigned* err) {
    mbar_arrive(bar);
    const bool ok = mbar_wait(bar, phase, abort, err);
    phase ^= 1u;
    return ok;
}

// Bounded wait that ignores the abort flag (used only while unwinding).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > 100000000ull) break;
    }
}

__global__ void __launch_bounds__(NTHREADS, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const Params P) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - smem_u32(smem_raw));
    const uint32_t s_ring = base;
    const uint32_t s_q = base + RING_BYTES;
    const uint32_t s_bars = s_q + Q_BYTES + XCH_BYTES;
    float* xch = reinterpret_cast<float*>(base_ptr + RING_BYTES + Q_BYTES);
    uint32_t* tmem_base_ptr =
        reinterpret_cast<uint32_t*>(base_ptr + RING_BYTES + Q_BYTES + XCH_BYTES + NUM_BARS * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_ptr + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(bar_full(s_bars, s), 1);
            mbar_init(bar_empty(s_bars, s), 1);
        }
        mbar_init(bar_qfull(s_bars), 1);
        mbar_init(bar_qempty(s_bars), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_sfull(s_bars, i), 1);
            mbar_init(bar_pfull(s_bars, i), NSOFT);
        }
        mbar_init(bar_ofull(s_bars), 1);
        mbar_init(bar_drain(s_bars), 1);
        mbar_init(bar_group(s_bars), NSOFT);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_base_ptr), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_ptr;

    SegIter it;
    it.init(P, blockIdx.x);
    int qt, jb, je, n;
    bool is_first;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t ring = 0;
            int seg = 0;
            bool ok = true;
            auto acquire = [&](uint32_t& slot_addr) -> int {
                const int slot = ring % NSLOT;
                const uint32_t ph = (ring / NSLOT) & 1u;
                if (!mbar_wait(bar_empty(s_bars, slot), ph ^ 1u, abort_flag, P.err)) return -1;
                slot_addr = s_ring + slot * SLOT_BYTES;
                return slot;
            };
            auto load_k = [&](int j) -> bool {
                for (int c = 0; c < 4; ++c) {
                    uint32_t dst;
                    const int slot = acquire(dst);
                    if (slot < 0) return false;
                    mbar_arrive_expect_tx(bar_full(s_bars, slot), SLOT_BYTES);
                    tma_load_2d(dst, &tm_k, bar_full(s_bars, slot), c * 64, j * BN);
                    ++ring;
                }
                return true;
            };
            auto load_v = [&](int j) -> bool {
                for (int sub = 0; sub < 4; ++sub) {
                    uint32_t dst;
                    const int slot = acquire(dst);
                    if (slot < 0) return false;
                    mbar_arrive_expect_tx(bar_full(s_bars, slot), SLOT_BYTES);
                    for (int c = 0; c < 4; ++c)
                        tma_load_2d(dst + c * 4096, &tm_v, bar_full(s_bars, slot), c * 64,
                                    j * BN + sub * 32);
                    ++ring;
                }
                return true;
            };
            while (ok && it.next(P, qt, jb, je, n, is_first)) {
                if (!mbar_wait(bar_qempty(s_bars), (seg & 1) ^ 1, abort_flag, P.err)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(bar_qfull(s_bars), Q_BYTES);
                for (int c = 0; c < 4; ++c)
                    tma_load_2d(s_q + c * (BM * 128), &tm_q, bar_qfull(s_bars), c * 64, qt * BM);
                ok = load_k(jb);
                for (int j = jb; ok && j < je; ++j) {
                    if (j + 1 < je) ok = load_k(j + 1);
                    if (ok) ok = load_v(j);
                }
                ++seg;
            }
            if (!ok) {
                // Unwind: let every copy still in flight land before the CTA exits.
                for (int s = 0; s < NSLOT; ++s) {
                    const uint32_t fills = ring > (uint32_t)s ? (ring - s + NSLOT - 1) / NSLOT : 0;
                    if (fills) drain_wait(bar_full(s_bars, s), (fills - 1) & 1u);
                }
                if (seg > 0) drain_wait(bar_qfull(s_bars), (seg - 1) & 1);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t ring = 0;
            uint32_t g = 0;
            int seg = 0;
            bool ok = true;
            auto take = [&](int& slot) -> bool {
                slot = ring % NSLOT;
                const uint32_t ph = (ring / NSLOT) & 1u;
                if (!mbar_wait(bar_full(s_bars, slot), ph, abort_flag, P.err)) return false;
                tc_fence_after();
                return true;
            };
            auto issue_qk = [&](uint32_t s_col) -> bool {
                for (int c = 0; c < 4; ++c) {
                    int slot;
                    if (!take(slot)) return false;
                    const uint32_t kaddr = s_ring + slot * SLOT_BYTES;
                    const uint32_t qaddr = s_q + c * (BM * 128);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t a = sdesc_sw128(qaddr + kk * 32, 16, 1024);
                        const uint64_t b = sdesc_sw128(kaddr + kk * 32, 16, 1024);
                        umma_ss(tmem + s_col, a, b, IDESC_QK, (c | kk) != 0);
                    }
                    umma_commit(bar_empty(s_bars, slot));
                    ++ring;
                }
                return true;
            };
            auto issue_pv = [&](uint32_t s_col, bool acc0) -> bool {
                for (int sub = 0; sub < 4; ++sub) {
                    int slot;
                    if (!take(slot)) return false;
                    const uint32_t vaddr = s_ring + slot * SLOT_BYTES;
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        const uint64_t b = sdesc_sw128(vaddr + ks * 2048, 4096, 1024);
                        // P of keys kb .. kb + 15: half kb / 64 sits at columns
                        // 64 (kb / 64) + (kb % 64) / 2 of the S buffer.
                        const int kb = sub * 32 + ks * 16;
                        const uint32_t a_tmem = tmem + s_col + (kb >> 6) * 64 + ((kb & 63) >> 1);
                        umma_ts(tmem + O_COL, a_tmem, b, IDESC_PV, (acc0 || sub || ks) ? 1u : 0u);
                    }
                    umma_commit(bar_empty(s_bars, slot));
                    ++ring;
                }
                return true;
            };
            while (ok && it.next(P, qt, jb, je, n, is_first)) {
                if (!mbar_wait(bar_qfull(s_bars), seg & 1, abort_flag, P.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                ok = issue_qk(S_COL0 + (g & 1) * BN);
                if (!ok) break;
                umma_commit(bar_sfull(s_bars, g & 1));
                if (je - jb == 1) umma_commit(bar_qempty(s_bars));
                for (int j = jb; j < je; ++j) {
                    const uint32_t gg = g + (j - jb);
                    if (j + 1 < je) {
                        ok = issue_qk(S_COL0 + ((gg + 1) & 1) * BN);
                        if (!ok) break;
                        umma_commit(bar_sfull(s_bars, (gg + 1) & 1));
                        if (j + 1 == je - 1) umma_commit(bar_qempty(s_bars));
                    }
                    if (!mbar_wait(bar_pfull(s_bars, gg & 1), (gg >> 1) & 1, abort_flag, P.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    ok = issue_pv(S_COL0 + (gg & 1) * BN, j > jb);
                    if (!ok) break;
                    umma_commit(bar_ofull(s_bars));
                }
                g += je - jb;
                ++seg;
            }
            if (!ok) {
                // Unwind: wait for every UMMA already issued before TMEM is freed.
                umma_commit(bar_drain(s_bars));
                drain_wait(bar_drain(s_bars), 0);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax / epilogue
        // Warpgroup hg owns S columns [64 hg, 64 hg + 64) of every tile and O
        // columns [128 hg, 128 hg + 128).  Row maxima: each thread writes its
        // half maximum to xch[tile parity][hg][row]; after the group barrier it
        // reads its partner's, so both threads of a row see the same maximum.
        const int hg = (warp - 2) >> 2;
        const int wq = warp & 3;           // TMEM lane quarter this warp may access
        const int row = wq * 32 + lane;    // tile row == TMEM lane
        const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
        float* xl = xch + 4 * BM;          // row-sum halves [hg][row]
        const uint32_t gbar = bar_group(s_bars);
        uint32_t gphase = 0;
        const float sl2 = P.scale_log2;
        uint32_t g = 0;
        bool ok = true;
        while (ok && it.next(P, qt, jb, je, n, is_first)) {
            const int m_row = qt * BM + row;
            const bool valid = m_row < P.M_total;
            const int lim = P.KV - P.Q + m_row / HQ;           // last visible key
            const int j_mask = (P.KV - P.Q + (qt * BM) / HQ + 1) / BN;  // first tile to mask
            float m_ref = -INFINITY;
            float l = 0.f;
            for (int j = jb; j < je; ++j) {
                const uint32_t gg = g + (j - jb);
                const uint32_t s_col = S_COL0 + (gg & 1) * BN;
                ok = mbar_wait(bar_sfull(s_bars, gg & 1), (gg >> 1) & 1, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                uint32_t sr[BN / 2];
#pragma unroll
                for (int c = 0; c < BN / 64; ++c)
                    tmem_ld32(t_lane + s_col + 64 * hg + 32 * c,
                              *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
                tmem_ld_wait<BN / 2>(sr);
                float* s = reinterpret_cast<float*>(sr);
                if (j >= j_mask) {
                    const int k0 = j * BN + 64 * hg;
#pragma unroll
                    for (int c = 0; c < BN / 2; ++c)
                        if (k0 + c > lim) s[c] = -INFINITY;
                }
                float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
                for (int c = 4; c < BN / 2; c += 4) {
                    mx0 = fmaxf(mx0, s[c]);
                    mx1 = fmaxf(mx1, s[c + 1]);
                    mx2 = fmaxf(mx2, s[c + 2]);
                    mx3 = fmaxf(mx3, s[c + 3]);
                }
                const float hm = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
                float* xp = xch + (gg & 1) * (2 * BM);
                xp[hg * BM + row] = hm;
                ok = group_sync(gbar, gphase, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                const float mx = fmaxf(xp[row], xp[BM + row]) * sl2;
                bool o_seen = false;
                if (j == jb) {
                    m_ref = mx;
                } else {
                    const bool need = mx > m_ref + RESCALE_THRESHOLD;
                    if (__any_sync(0xffffffffu, need)) {
                        ok = mbar_wait(bar_ofull(s_bars), (gg - 1) & 1, abort_flag, P.err);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                        tc_fence_after();
                        o_seen = true;
                        const float f = need ? ex2(m_ref - mx) : 1.0f;
                        if (need) {
                            l *= f;
                            m_ref = mx;
                        }
#pragma unroll 1
                        for (int c = 0; c < D / 64; ++c) {
                            uint32_t o[32];
                            const uint32_t oc = O_COL + 128 * hg + 32 * c;
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
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
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
                tmem_st32(t_lane + s_col + 64 * hg, pk);
                l += (l0 + l1) + (l2 + l3);
                tmem_st_wait();
                if (j > jb && !o_seen) {
                    ok = mbar_wait(bar_ofull(s_bars), (gg - 1) & 1, abort_flag, P.err);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                }
                tc_fence_before();
                mbar_arrive(bar_pfull(s_bars, gg & 1));
            }
            if (!ok) break;
            // ---------------------------------------------------------- epilogue
            const uint32_t gl = g + (je - jb) - 1;
            ok = mbar_wait(bar_ofull(s_bars), gl & 1, abort_flag, P.err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            // Row sum: the two halves, added in a fixed order.
            xl[hg * BM + row] = l;
            ok = group_sync(gbar, gphase, abort_flag, P.err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const float l_row = xl[row] + xl[BM + row];
            if (jb == 0 && je == n) {
                const float inv = (l_row > 0.f) ? 1.0f / l_row : 0.f;
                uint4* dst = reinterpret_cast<uint4*>(P.out + (size_t)m_row * D + 128 * hg);
#pragma unroll 1
                for (int c = 0; c < D / 64; ++c) {
                    uint32_t o[32];
                    tmem_ld32(t_lane + O_COL + 128 * hg + 32 * c, o);
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
                const size_t prow = ((size_t)blockIdx.x * 2 + slot) * BM + row;
                uint4* dst = reinterpret_cast<uint4*>(P.ws_o + prow * D + 128 * hg);
#pragma unroll 1
                for (int c = 0; c < D / 64; ++c) {
                    uint32_t o[32];
                    tmem_ld32(t_lane + O_COL + 128 * hg + 32 * c, o);
                    tmem_ld_wait<32>(o);
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

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// A q-tile cut between CTAs c0 .. c_last: its first piece is CTA c0's last
// segment (partial slot slot0), the others are the first segments (slot 0) of
// CTAs c0 + 1 .. c_last.  Found on the host from the same shape-only schedule.
constexpr int kMaxCtas = 160;
struct MergeTasks {
    int n;
    int4 task[kMaxCtas];  // (q-tile, c0, slot0, c_last)
};

// blockIdx.x picks a cut q-tile, blockIdx.y 8 of its 128 rows; thread
// (row, lane) merges 8 consecutive d.  Pieces are combined in CTA order (exact
// log-sum-exp merge), so the result does not depend on timing.
__global__ void __launch_bounds__(256)
prefill_merge_kernel(const Params P, const __grid_constant__ MergeTasks T) {
    const int4 tk = T.task[blockIdx.x];
    const int t = tk.x, c0 = tk.y, slot0 = tk.z, c_last = tk.w;
    const int r = blockIdx.y * 8 + (threadIdx.x >> 5);
    const int m_row = t * BM + r;
    if (m_row >= P.M_total) return;
    const int d0 = (threadIdx.x & 31) * 8;
    float M = -INFINITY;
    for (int c = c0; c <= c_last; ++c) {
        const size_t prow = ((size_t)c * 2 + (c == c0 ? slot0 : 0)) * BM + r;
        M = fmaxf(M, P.ws_ml[prow * 2]);
    }
    float L = 0.f;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int c = c0; c <= c_last; ++c) {
        const size_t prow = ((size_t)c * 2 + (c == c0 ? slot0 : 0)) * BM + r;
        const float mp = P.ws_ml[prow * 2];
        const float w = (mp == -INFINITY) ? 0.f : exp2f(mp - M);
        L += P.ws_ml[prow * 2 + 1] * w;
        const float4* o = reinterpret_cast<const float4*>(P.ws_o + prow * D + d0);
        const float4 a = o[0], b = o[1];
        acc[0] += a.x * w; acc[1] += a.y * w; acc[2] += a.z * w; acc[3] += a.w * w;
        acc[4] += b.x * w; acc[5] += b.y * w; acc[6] += b.z * w; acc[7] += b.w * w;
    }
    const float inv = L > 0.f ? 1.0f / L : 0.f;
    uint4 hv = make_uint4(pack_half2(acc[0] * inv, acc[1] * inv), pack_half2(acc[2] * inv, acc[3] * inv),
                          pack_half2(acc[4] * inv, acc[5] * inv), pack_half2(acc[6] * inv, acc[7] * inv));
    *reinterpret_cast<uint4*>(P.out + (size_t)m_row * D + d0) = hv;
}

// Host side of the schedule: the cut q-tiles and their pieces.
static void find_cut_tiles(const Params& P, MergeTasks& T) {
    T.n = 0;
    long long cum = 0;
    int c = 0;  // first CTA whose range ends after cum
    for (int t = 0; t < P.num_qtiles; ++t) {
        const int n = kv_tiles(t, P.Q, P.KV, P.M_total);
        const long long t_end = cum + n;
        // CTA holding the tile's first iteration
        while (c + 1 < P.G && cta_begin(P.total, P.G, c + 1) <= cum) ++c;
        if (cta_begin(P.total, P.G, c + 1) < t_end) {  // the tile continues past CTA c
            int c_last = c + 1;
            while (c_last + 1 < P.G && cta_begin(P.total, P.G, c_last + 1) < t_end) ++c_last;
            const int slot0 = (cta_begin(P.total, P.G, c) == cum) ? 0 : 1;
            T.task[T.n++] = make_int4(t, c, slot0, c_last);
        }
        cum = t_end;
    }
}

}  // namespace prefill

size_t prefill_workspace_bytes(int Q, int KV, int num_sms) {
    (void)Q;
    (void)KV;
    const size_t per_cta = (size_t)2 * prefill::BM * (prefill::D + 2) * sizeof(float);
    return kWorkspaceCounterBytes + per_cta * (size_t)num_sms + 256;
}

int prefill_launch(const void* q, const void* k, const void* v, void* out, int Q, int KV,
                   float scale, cudaStream_t stream) {
    using namespace prefill;
    const DeviceInfo* di = device_info();
    if (!di) return GQA_ERR_CUDA;
    Params P;
    P.Q = Q;
    P.KV = KV;
    P.M_total = Q * HQ;
    P.num_qtiles = (P.M_total + BM - 1) / BM;
    long long total = 0;
    for (int t = 0; t < P.num_qtiles; ++t) total += kv_tiles(t, Q, KV, P.M_total);
    P.total = total;
    P.G = (int)(total < di->num_sms ? total : di->num_sms);
    if (P.G > kMaxCtas) P.G = kMaxCtas;
    P.scale_log2 = scale * 1.4426950408889634f;
    P.out = static_cast<__half*>(out);
    P.err = di->err_word;

    void* ws;
    size_t ws_bytes;
    current_workspace(&ws, &ws_bytes);
    const size_t need = kWorkspaceCounterBytes + (size_t)P.G * 2 * BM * (D + 2) * sizeof(float);
    if (P.G > 1 && (!ws || ws_bytes < need)) return GQA_ERR_WORKSPACE;
    if (ws) {
        float* w = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kWorkspaceCounterBytes);
        P.ws_o = w;
        P.ws_ml = w + (size_t)P.G * 2 * BM * D;
    } else {
        P.ws_o = nullptr;
        P.ws_ml = nullptr;
    }

    CUtensorMap tq, tk, tv;
    if (!make_map_2d_f16(&tq, q, (uint64_t)P.M_total, D, BM, 64) ||
        !make_map_2d_f16(&tk, k, (uint64_t)KV, D, BN, 64) ||
        !make_map_2d_f16(&tv, v, (uint64_t)KV, D, 32, 64))
        return GQA_ERR_CUDA;

    static bool attr_done[64] = {false};
    if (di->device < 64 && !attr_done[di->device]) {
        if (cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_BYTES) != cudaSuccess)
            return GQA_ERR_CUDA;
        attr_done[di->device] = true;
    }
    prefill_kernel<<<P.G, NTHREADS, SMEM_BYTES, stream>>>(tq, tk, tv, P);
    if (cudaGetLastError() != cudaSuccess) return GQA_ERR_CUDA;
    MergeTasks tasks;  // passed to the merge kernel by value
    find_cut_tiles(P, tasks);
    if (tasks.n > 0) {
        prefill_merge_kernel<<<dim3(tasks.n, BM / 8), 256, 0, stream>>>(P, tasks);
        if (cudaGetLastError() != cudaSuccess) return GQA_ERR_CUDA;
    }
    return GQA_OK;
}

}  // namespace gqa
