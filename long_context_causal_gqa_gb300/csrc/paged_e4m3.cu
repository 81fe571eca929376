// paged_e4m3.cu -- causal GQA verifier tail over an FP8-E4M3 paged KV cache.
//
// Problem ("[Perf] Ship the qualified SM70 long-context layout and drop its
// context fences", What / Changes): R <= 8 query rows (6R packed rows, Hq=6
// sharing Hkv=1) at the end of a context of up to 262144 keys; K and V are
// E4M3 bytes (one fp32 scale each) in page-16 blocks addressed through a
// block table of physical page ids; FP32 accumulation.  The page's operator
// decodes E4M3 through a shared lookup table and specialises the 8-row case;
// here the work is HBM-bound (one byte per K/V element) and shaped for sm_103a:
//
// * Split-KV: the context is cut into 128-key tiles (8 pages) and the tiles
//   into one contiguous range per SM.  Each split writes an (O, m, l) partial;
//   a merge kernel combines them in split order (exact log-sum-exp merge).
// * Swap-AB UMMA: keys are the M=128 dimension, the packed query rows the N
//   dimension (padded to NP = 16/32/48), so few rows waste no tensor work.
//     S^T[128 keys x NP] = K[128 x 256] . Q^T          (A = K in tensor memory)
//     O^T[256 d x NP]   += V^T[256 x 128] . P^T[128 x NP] (two M=128 halves)
// * E4M3 -> fp16 is pure bit work: fp16 bits = sign << 15 | (b & 0x7F) << 7
//   equals the E4M3 value times 2^-8 for every finite code (normal and
//   subnormal), so the 2^8 is folded into the K and V scales.  K is decoded by
//   the thread that owns its TMEM lane and stored as the UMMA A operand; V is
//   decoded into a 128B-swizzled fp16 smem tile.  Raw pages arrive by TMA
//   tensor copies (128-byte swizzle, so every thread reads its own key's row
//   without bank conflicts) through a 3-stage ring.
// * Softmax over keys runs across TMEM lanes.  A per-row reference max moves
//   only when a score exceeds it by more than 8 (log2 units); the common case
//   is one threshold compare and a CTA-wide vote per tile, and the exact
//   cross-lane max is taken only on the first tile or when the vote fires.
//   Row sums stay per thread until the split's end.
//
// Warp roles (320 threads): 0 bulk-copy producer, 1 TMEM owner + UMMA issuer,
// 2..5 "key" warps (K decode, softmax, epilogue; thread = TMEM lane),
// 6..9 V decode warps.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"
#include "sm100.cuh"

namespace gqa {
namespace paged {

constexpr int D = kHeadDim;      // 256
constexpr int HQ = kHq;          // 6
constexpr int PAGE = kPage;      // 16 tokens
constexpr int TILE = 128;        // keys per tile
constexpr int PAGES_PER_TILE = TILE / PAGE;
constexpr int PAGE_BYTES = PAGE * D;            // 4096 (Hkv = 1, one byte per element)
constexpr int RAW_STAGE = TILE * D;             // 32 KB of E4M3 per K or V tile
constexpr int NRAW = 3;
constexpr int V_BYTES = TILE * D * 2;           // fp16 V tile, 64 KB
constexpr int NTHREADS = 320;
constexpr float RESCALE_THRESHOLD = 8.0f;

struct Params {
    const uint8_t* kcache;
    const uint8_t* vcache;
    const float* kscale;
    const float* vscale;
    const int32_t* table;
    const __half* q;
    int num_pages, ctx_len, R, nq, n_tiles, G;
    float scale;
    float* ws_o;    // [G][nq][D] unnormalised partial O (in units of the fp16 V)
    float* ws_ml;   // [G][nq][2]  (m in log2 units, l)
    __half* out;
    unsigned* err;
};

template <int NP>
struct Layout {
    static constexpr int Q_BYTES = NP * D * 2;       // 4 chunks [NP][64] fp16
    static constexpr int PT_BYTES = NP * TILE * 2;   // 2 chunks [NP][64 keys] fp16
    static constexpr int OFF_V = 0;
    static constexpr int OFF_RAW = OFF_V + V_BYTES;
    static constexpr int OFF_Q = OFF_RAW + NRAW * RAW_STAGE;
    static constexpr int OFF_PT = OFF_Q + Q_BYTES;
    static constexpr int OFF_RED = OFF_PT + 2 * PT_BYTES;       // [4][NP] floats
    static constexpr int OFF_MREF = OFF_RED + 4 * NP * 4;        // [NP] floats
    static constexpr int OFF_FAC = OFF_MREF + NP * 4;            // [NP] floats
    static constexpr int OFF_FLAG = OFF_FAC + NP * 4;            // [2][4] ints
    static constexpr int OFF_BAR = (OFF_FLAG + 32 + 7) & ~7;
    static constexpr int NUM_BARS = 2 * NRAW + 12;
    static constexpr int OFF_TMEM = OFF_BAR + NUM_BARS * 8;
    static constexpr int BYTES = OFF_TMEM + 16;
    static constexpr int SMEM = BYTES + 1024;
    // TMEM columns
    static constexpr uint32_t K_COL = 0;             // 2 x 128 (fp16 pairs)
    static constexpr uint32_t S_COL = 256;           // 2 x NP
    static constexpr uint32_t O_COL = 256 + 2 * NP;  // 2 halves x NP
};

// mbarrier indices
enum {
    B_RAW_FULL = 0,          // [NRAW]
    B_RAW_EMPTY = NRAW,      // [NRAW]
    B_K_READY = 2 * NRAW,    // [2]
    B_S_FULL = 2 * NRAW + 2, // [2]
    B_P_READY = 2 * NRAW + 4,// [2]
    B_PT_EMPTY = 2 * NRAW + 6, // [2] PV of that P^T buffer done
    B_V_READY = 2 * NRAW + 8,
    B_V_EMPTY = 2 * NRAW + 9,
    B_DRAIN = 2 * NRAW + 10,
    B_GROUP = 2 * NRAW + 11,  // key-thread group barrier
};

// 4 E4M3 bytes -> 4 fp16 (value * 2^-8) as two half2 words.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t x, uint32_t& lo, uint32_t& hi) {
    const uint32_t a = __byte_perm(x, 0u, 0x1404);  // [0, b0, 0, b1]
    const uint32_t b = __byte_perm(x, 0u, 0x3424);  // [0, b2, 0, b3]
    lo = (a & 0x80008000u) | ((a >> 1) & 0x3F803F80u);
    hi = (b & 0x80008000u) | ((b >> 1) & 0x3F803F80u);
}

// Byte offset of 16-byte unit u (0..7) of row r inside a 128B-swizzled block.
__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t u) {
    return r * 128u + ((u ^ (r & 7u)) << 4);
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > 100000000ull) break;
    }
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

template <int NP>
__global__ void __launch_bounds__(NTHREADS, 1)
paged_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const Params P) {
    using L = Layout<NP>;
    constexpr uint32_t IDESC_QK = idesc_f16_f32(128, NP, false, false);
    constexpr uint32_t IDESC_PV = idesc_f16_f32(128, NP, true, false);

    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (sbase - smem_u32(smem_raw));
    const uint32_t s_v = sbase + L::OFF_V;
    const uint32_t s_raw = sbase + L::OFF_RAW;
    const uint32_t s_q = sbase + L::OFF_Q;
    const uint32_t s_pt = sbase + L::OFF_PT;
    float* red = reinterpret_cast<float*>(gbase + L::OFF_RED);
    float* mref = reinterpret_cast<float*>(gbase + L::OFF_MREF);
    float* fac = reinterpret_cast<float*>(gbase + L::OFF_FAC);
    volatile int* flags = reinterpret_cast<volatile int*>(gbase + L::OFF_FLAG);
    const uint32_t bars = sbase + L::OFF_BAR;
    uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(gbase + L::OFF_TMEM);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_ptr + 1);
    auto bar = [&](int i) { return bars + 8u * i; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int split = blockIdx.x;
    const int t_begin = (int)((long long)split * P.n_tiles / P.G);
    const int t_end = (int)((long long)(split + 1) * P.n_tiles / P.G);
    const int ntl = t_end - t_begin;
    const int n_logical = (P.ctx_len + PAGE - 1) / PAGE;

    // ---- set-up: barriers, Q -> smem (swizzled, zero padding rows), TMEM
    if (threadIdx.x == 0) {
        for (int s = 0; s < NRAW; ++s) {
            mbar_init(bar(B_RAW_FULL + s), 1);
            mbar_init(bar(B_RAW_EMPTY + s), 128);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_K_READY + b), 128);
            mbar_init(bar(B_S_FULL + b), 1);
            mbar_init(bar(B_P_READY + b), 128);
            mbar_init(bar(B_PT_EMPTY + b), 1);
        }
        mbar_init(bar(B_V_READY), 128);
        mbar_init(bar(B_V_EMPTY), 1);
        mbar_init(bar(B_DRAIN), 1);
        mbar_init(bar(B_GROUP), 128);
        *abort_flag = 0;
        fence_mbar_init();
    }
    for (int u = threadIdx.x; u < NP * (D / 8); u += NTHREADS) {
        const int r = u / (D / 8);          // packed query row
        const int c16 = u % (D / 8);        // 16-byte unit along d
        uint4 val = make_uint4(0, 0, 0, 0);
        if (r < P.nq) val = *reinterpret_cast<const uint4*>(P.q + (size_t)r * D + c16 * 8);
        const uint32_t dst = s_q + (c16 / 8) * (NP * 128) + sw128(r, c16 % 8);
        *reinterpret_cast<uint4*>(gbase + L::OFF_Q + (dst - s_q)) = val;
    }
    for (int c = threadIdx.x; c < NP; c += NTHREADS) mref[c] = -INFINITY;
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_ptr), 512);
        tmem_relinquish();
    }
    fence_async_shared();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_ptr;
    const float kscale = *P.kscale;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && ntl > 0) {
            uint32_t item = 0;
            bool ok = true;
            for (int jj = 0; jj < ntl && ok; ++jj) {
                const int tile = t_begin + jj;
                const int p0 = tile * PAGES_PER_TILE;
                int phys[PAGES_PER_TILE];
                int npg = 0;
#pragma unroll
                for (int p = 0; p < PAGES_PER_TILE; ++p) {
                    int id = 0;
                    if (p0 + p < n_logical) {
                        id = __ldg(P.table + p0 + p);
                        if (id < 0 || id >= P.num_pages) {
                            atomicOr(P.err, kErrBadPageId);
                            id = 0;
                        }
                        npg = p + 1;
                    }
                    phys[p] = id;
                }
                for (int kv = 0; kv < 2 && ok; ++kv) {
                    const int s = item % NRAW;
                    const uint32_t ph = (item / NRAW) & 1u;
                    if (!mbar_wait(bar(B_RAW_EMPTY + s), ph ^ 1u, abort_flag, P.err)) {
                        ok = false;
                        break;
                    }
                    const CUtensorMap* tm = kv == 0 ? &tm_k : &tm_v;
                    mbar_arrive_expect_tx(bar(B_RAW_FULL + s), npg * PAGE_BYTES);
                    // Stage layout: [2 halves of d][128 keys][128 B], 128B-swizzled.
                    for (int p = 0; p < npg; ++p)
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            tma_load_2d(s_raw + s * RAW_STAGE + h * (TILE * 128) + p * (PAGE * 128),
                                        tm, bar(B_RAW_FULL + s), h * 128, phys[p] * PAGE);
                    ++item;
                }
            }
            if (!ok) {
                for (int s = 0; s < NRAW; ++s) {
                    const uint32_t fills = item > (uint32_t)s ? (item - s + NRAW - 1) / NRAW : 0;
                    if (fills) drain_wait(bar(B_RAW_FULL + s), (fills - 1) & 1u);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ UMMA issuer
        if (lane == 0 && ntl > 0) {
            bool ok = true;
            auto issue_pv = [&](int x) -> bool {
                if (!mbar_wait(bar(B_P_READY + (x & 1)), (x >> 1) & 1, abort_flag, P.err))
                    return false;
                if (!mbar_wait(bar(B_V_READY), x & 1, abort_flag, P.err)) return false;
                tc_fence_after();
                const uint32_t pt = s_pt + (x & 1) * L::PT_BYTES;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
#pragma unroll
                    for (int ks = 0; ks < TILE / 16; ++ks) {
                        const uint64_t a = sdesc_sw128(s_v + (2 * h) * (TILE * 128) + ks * 2048,
                                                       TILE * 128, 1024);
                        const uint64_t b =
                            sdesc_sw128(pt + (ks / 4) * (NP * 128) + (ks % 4) * 32, 16, 1024);
                        umma_ss(tmem + L::O_COL + h * NP, a, b, IDESC_PV, (x > 0 || ks > 0));
                    }
                }
                umma_commit(bar(B_PT_EMPTY + (x & 1)));
                umma_commit(bar(B_V_EMPTY));
                return true;
            };
            for (int jj = 0; jj < ntl && ok; ++jj) {
                const int b = jj & 1;
                if (!mbar_wait(bar(B_K_READY + b), (jj >> 1) & 1, abort_flag, P.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t bq =
                        sdesc_sw128(s_q + (kk / 4) * (NP * 128) + (kk % 4) * 32, 16, 1024);
                    umma_ts(tmem + L::S_COL + b * NP, tmem + L::K_COL + b * 128 + kk * 8, bq,
                            IDESC_QK, kk > 0);
                }
                umma_commit(bar(B_S_FULL + b));
                if (jj >= 1) ok = issue_pv(jj - 1);
            }
            if (ok) ok = issue_pv(ntl - 1);
            if (!ok) {
                umma_commit(bar(B_DRAIN));
                drain_wait(bar(B_DRAIN), 0);
            }
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------ key warps
        const int wq = warp & 3;
        const int k = wq * 32 + lane;                       // TMEM lane = key in tile = d in O^T half
        const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
        const float sl2 = P.scale * kscale * 256.0f * 1.4426950408889634f;
        const int lim_base = P.ctx_len - P.R;               // row r sees keys <= lim_base + r
        float lpart[NP];
#pragma unroll
        for (int c = 0; c < NP; ++c) lpart[c] = 0.f;
        uint32_t raw_item = 0;
        uint32_t gphase = 0;
        bool ok = ntl > 0;

        // Decode tile jj's K (raw stage) into TMEM K buffer jj & 1.
        auto decode_k = [&](int jj) -> bool {
            const int s = raw_item % NRAW;
            const uint32_t ph = (raw_item / NRAW) & 1u;
            if (!mbar_wait(bar(B_RAW_FULL + s), ph, abort_flag, P.err)) return false;
            const int key = (t_begin + jj) * TILE + k;
            const bool live = key / PAGE < n_logical;   // page loaded (else stale smem)
            const uint8_t* src = gbase + L::OFF_RAW + s * RAW_STAGE + k * 128;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t w[64];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    uint4 x = make_uint4(0, 0, 0, 0);
                    if (live)
                        x = *reinterpret_cast<const uint4*>(src + half * (TILE * 128) +
                                                            ((i ^ (k & 7)) << 4));
                    e4m3x4_to_f16(x.x, w[8 * i + 0], w[8 * i + 1]);
                    e4m3x4_to_f16(x.y, w[8 * i + 2], w[8 * i + 3]);
                    e4m3x4_to_f16(x.z, w[8 * i + 4], w[8 * i + 5]);
                    e4m3x4_to_f16(x.w, w[8 * i + 6], w[8 * i + 7]);
                }
                tmem_st32(t_lane + L::K_COL + (jj & 1) * 128 + half * 64, w);
                tmem_st32(t_lane + L::K_COL + (jj & 1) * 128 + half * 64 + 32, w + 32);
            }
            tmem_st_wait();
            mbar_arrive(bar(B_RAW_EMPTY + s));
            raw_item += 2;  // skip the V stage of this tile
            tc_fence_before();
            mbar_arrive(bar(B_K_READY + (jj & 1)));
            return true;
        };

        if (ok) ok = decode_k(0);
        for (int jj = 0; jj < ntl && ok; ++jj) {
            if (jj + 1 < ntl) {
                ok = decode_k(jj + 1);
                if (!ok) break;
            }
            const int b = jj & 1;
            ok = mbar_wait(bar(B_S_FULL + b), (jj >> 1) & 1, abort_flag, P.err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            float s[NP];
            {
                uint32_t r[NP];
#pragma unroll
                for (int c = 0; c < NP; c += 16) tmem_ld16(t_lane + L::S_COL + b * NP + c, r + c);
                tmem_ld_wait<NP>(r);
#pragma unroll
                for (int c = 0; c < NP; ++c) s[c] = __uint_as_float(r[c]) * sl2;
            }
            const int key = (t_begin + jj) * TILE + k;
            if ((t_begin + jj) * TILE + TILE - 1 > lim_base) {
#pragma unroll
                for (int c = 0; c < NP; ++c) {
                    const int r = c / HQ;
                    const bool vis = (c < P.nq) ? (key <= lim_base + r) : (key < P.ctx_len);
                    if (!vis) s[c] = -INFINITY;
                }
            }
            // Vote: does any score exceed its row's reference max by > threshold?
            bool exceed = false;
#pragma unroll
            for (int c = 0; c < NP; ++c) exceed |= s[c] > mref[c] + RESCALE_THRESHOLD;
            const unsigned vote = __ballot_sync(0xffffffffu, exceed);
            volatile int* fl = flags + (jj & 1) * 4;
            if (lane == 0) fl[wq] = vote != 0;
            ok = group_sync(bar(B_GROUP), gphase, abort_flag, P.err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const bool any = fl[0] | fl[1] | fl[2] | fl[3];
            if (any) {
                // Exact column max over the 128 keys of this tile.
#pragma unroll
                for (int c = 0; c < NP; ++c) {
                    float m = s[c];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                    if (lane == 0) red[wq * NP + c] = m;
                }
                ok = group_sync(bar(B_GROUP), gphase, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                if (k < NP) {
                    const int c = k;
                    const float tmax = fmaxf(fmaxf(red[c], red[NP + c]),
                                             fmaxf(red[2 * NP + c], red[3 * NP + c]));
                    const float old = mref[c];
                    float f = 1.0f;
                    if (tmax > old + RESCALE_THRESHOLD) {
                        f = (old == -INFINITY) ? 0.f : ex2(old - tmax);
                        mref[c] = tmax;
                    }
                    fac[c] = f;
                }
                ok = group_sync(bar(B_GROUP), gphase, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                if (jj > 0) {
                    // O^T must hold every earlier P.V before it is rescaled.
                    const int x = jj - 1;
                    ok = mbar_wait(bar(B_PT_EMPTY + (x & 1)), (x >> 1) & 1, abort_flag, P.err);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t r[NP];
#pragma unroll
                        for (int c = 0; c < NP; c += 16)
                            tmem_ld16(t_lane + L::O_COL + h * NP + c, r + c);
                        tmem_ld_wait<NP>(r);
#pragma unroll
                        for (int c = 0; c < NP; ++c)
                            r[c] = __float_as_uint(__uint_as_float(r[c]) * fac[c]);
#pragma unroll
                        for (int c = 0; c < NP; c += 16)
                            tmem_st16(t_lane + L::O_COL + h * NP + c, r + c);
                    }
                    tmem_st_wait();
                }
#pragma unroll
                for (int c = 0; c < NP; ++c) lpart[c] *= fac[c];
            }
            // P^T buffer b is free once the P.V two tiles back has completed.
            ok = mbar_wait(bar(B_PT_EMPTY + b), ((jj >> 1) & 1) ^ 1, abort_flag, P.err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            uint8_t* pt = gbase + L::OFF_PT + b * L::PT_BYTES;
            const int kc = k >> 6;          // 64-key chunk
            const int kin = k & 63;
#pragma unroll
            for (int c = 0; c < NP; ++c) {
                const float m = mref[c];
                const float p = ex2(s[c] - (m == -INFINITY ? 0.f : m));
                lpart[c] += p;
                const uint32_t off = kc * (NP * 128) + sw128(c, kin >> 3) + (kin & 7) * 2;
                *reinterpret_cast<__half*>(pt + off) = __float2half_rn(p);
            }
            fence_async_shared();
            mbar_arrive(bar(B_P_READY + b));
        }
        // ---------------------------------------------------------- epilogue
        if (ok && ntl > 0) {
            const int x = ntl - 1;
            ok = mbar_wait(bar(B_PT_EMPTY + (x & 1)), (x >> 1) & 1, abort_flag, P.err);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok && ntl > 0) {
            tc_fence_after();
            // Row sums: reduce the per-thread partial sums over the 128 keys.
#pragma unroll
            for (int c = 0; c < NP; ++c) {
                float v = lpart[c];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (lane == 0) red[wq * NP + c] = v;
            }
            ok = group_sync(bar(B_GROUP), gphase, abort_flag, P.err);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok && ntl > 0) {
            if (k < P.nq) {
                const int c = k;
                const float l = (red[c] + red[NP + c]) + (red[2 * NP + c] + red[3 * NP + c]);
                P.ws_ml[((size_t)split * P.nq + c) * 2 + 0] = mref[c];
                P.ws_ml[((size_t)split * P.nq + c) * 2 + 1] = l;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t r[NP];
#pragma unroll
                for (int c = 0; c < NP; c += 16) tmem_ld16(t_lane + L::O_COL + h * NP + c, r + c);
                tmem_ld_wait<NP>(r);
                const int d = h * 128 + k;
#pragma unroll
                for (int c = 0; c < NP; ++c)
                    if (c < P.nq) P.ws_o[((size_t)split * P.nq + c) * D + d] = __uint_as_float(r[c]);
            }
        }
    } else {
        // ------------------------------------------------------------ V decode warps
        const int t = threadIdx.x - 192;                 // 0..127
        uint32_t raw_item = 1;                           // V stages are the odd items
        bool ok = ntl > 0;
        for (int jj = 0; jj < ntl && ok; ++jj) {
            const int s = raw_item % NRAW;
            const uint32_t ph = (raw_item / NRAW) & 1u;
            ok = mbar_wait(bar(B_RAW_FULL + s), ph, abort_flag, P.err);
            if (!ok) break;
            ok = mbar_wait(bar(B_V_EMPTY), (jj & 1) ^ 1, abort_flag, P.err);
            if (!ok) break;
            const uint8_t* src = gbase + L::OFF_RAW + s * RAW_STAGE;
            const int tile_key0 = (t_begin + jj) * TILE;
            // 128 keys x 16 raw units of 16 bytes (16 d each); thread t handles
            // units t, t + 128, ...; 8 consecutive threads read one key's half row.
#pragma unroll 4
            for (int i = 0; i < 16; ++i) {
                const int unit = i * 128 + t;
                const int key = unit >> 4;        // 0..127
                const int u = unit & 15;          // d = 16u .. 16u + 15
                const int h = u >> 3;
                uint4 x = make_uint4(0, 0, 0, 0);
                if ((tile_key0 + key) / PAGE < n_logical)
                    x = *reinterpret_cast<const uint4*>(src + h * (TILE * 128) + key * 128 +
                                                        (((u & 7) ^ (key & 7)) << 4));
                uint32_t w[8];
                e4m3x4_to_f16(x.x, w[0], w[1]);
                e4m3x4_to_f16(x.y, w[2], w[3]);
                e4m3x4_to_f16(x.z, w[4], w[5]);
                e4m3x4_to_f16(x.w, w[6], w[7]);
                // fp16 tile: chunk u / 4 (64 d), 16-byte units 2(u%4), 2(u%4)+1
                const int chunk = u >> 2;
                const int uu = (u & 3) * 2;
                uint8_t* dst = gbase + L::OFF_V + chunk * (TILE * 128);
                *reinterpret_cast<uint4*>(dst + sw128(key, uu)) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4*>(dst + sw128(key, uu + 1)) =
                    make_uint4(w[4], w[5], w[6], w[7]);
            }
            fence_async_shared();
            mbar_arrive(bar(B_RAW_EMPTY + s));
            mbar_arrive(bar(B_V_READY));
            raw_item += 2;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// out[c, d] = vscale * 256 * sum_s w_s O_s[c, d] / sum_s w_s l_s, w_s = 2^(m_s - M).
// Block (c, dg) merges packed row c for d = 32 dg .. 32 dg + 31.  The split
// weights are computed once per block in shared memory; warp w then sums the
// splits s = w, w + 8, ... for its lane's d, and the eight warp sums are added
// in a fixed order, so the result does not depend on timing.
constexpr int MERGE_MAX_SPLITS = 1024;

__global__ void __launch_bounds__(256) paged_merge_kernel(const Params P) {
    __shared__ float w_s[MERGE_MAX_SPLITS];
    __shared__ float red[8][33];
    __shared__ float stat[2];
    const int c = blockIdx.x;
    const int d = blockIdx.y * 32 + (threadIdx.x & 31);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = P.G;
    // Phase 1: M = max_s m_s, w_s = 2^(m_s - M), L = sum_s w_s l_s.
    float mx = -INFINITY;
    for (int s = threadIdx.x; s < G; s += 256) {
        const float m = P.ws_ml[((size_t)s * P.nq + c) * 2];
        w_s[s] = m;
        mx = fmaxf(mx, m);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) red[warp][32] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        float M = red[0][32];
        for (int w = 1; w < 8; ++w) M = fmaxf(M, red[w][32]);
        stat[0] = M;
    }
    __syncthreads();
    const float M = stat[0];
    float lsum = 0.f;
    for (int s = threadIdx.x; s < G; s += 256) {
        const float m = w_s[s];
        const float w = (m == -INFINITY) ? 0.f : exp2f(m - M);
        w_s[s] = w;
        lsum += w * P.ws_ml[((size_t)s * P.nq + c) * 2 + 1];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    __syncthreads();
    if (lane == 0) red[warp][32] = lsum;
    __syncthreads();
    if (threadIdx.x == 0) {
        float L = 0.f;
        for (int w = 0; w < 8; ++w) L += red[w][32];
        stat[1] = L;
    }
    // Phase 2: weighted sum of the partial O over the splits.
    float acc = 0.f;
#pragma unroll 4
    for (int s = warp; s < G; s += 8) acc += w_s[s] * P.ws_o[((size_t)s * P.nq + c) * D + d];
    red[warp][lane] = acc;
    __syncthreads();
    if (warp == 0) {
        float a = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) a += red[w][lane];
        const float L = stat[1];
        const float vs = *P.vscale * 256.0f;
        P.out[(size_t)c * D + d] = __float2half_rn(L > 0.f ? a / L * vs : 0.f);
    }
}

template <int NP>
int launch_np(const CUtensorMap& tk, const CUtensorMap& tv, Params& P, cudaStream_t stream,
              int device) {
    using L = Layout<NP>;
    static bool attr_done[64] = {false};
    if (device < 64 && !attr_done[device]) {
        if (cudaFuncSetAttribute(paged_split_kernel<NP>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 L::SMEM) != cudaSuccess)
            return GQA_ERR_CUDA;
        attr_done[device] = true;
    }
    paged_split_kernel<NP><<<P.G, NTHREADS, L::SMEM, stream>>>(tk, tv, P);
    if (cudaGetLastError() != cudaSuccess) return GQA_ERR_CUDA;
    paged_merge_kernel<<<dim3(P.nq, D / 32), 256, 0, stream>>>(P);
    if (cudaGetLastError() != cudaSuccess) return GQA_ERR_CUDA;
    return GQA_OK;
}

}  // namespace paged

size_t paged_e4m3_workspace_bytes(int R, int ctx_len, int num_sms) {
    const int n_tiles = (ctx_len + paged::TILE - 1) / paged::TILE;
    const int G = n_tiles < num_sms ? n_tiles : num_sms;
    const size_t nq = (size_t)R * kHq;
    return kWorkspaceCounterBytes + (size_t)G * nq * (paged::D + 2) * sizeof(float) + 256;
}

int paged_e4m3_launch(const void* q, const uint8_t* kcache, const uint8_t* vcache,
                      const float* kscale, const float* vscale, const int32_t* block_table,
                      int num_pages, int ctx_len, int R, float scale, void* out,
                      cudaStream_t stream) {
    using namespace paged;
    const DeviceInfo* di = device_info();
    if (!di) return GQA_ERR_CUDA;
    Params P;
    P.kcache = kcache;
    P.vcache = vcache;
    P.kscale = kscale;
    P.vscale = vscale;
    P.table = block_table;
    P.q = static_cast<const __half*>(q);
    P.num_pages = num_pages;
    P.ctx_len = ctx_len;
    P.R = R;
    P.nq = R * HQ;
    P.n_tiles = (ctx_len + TILE - 1) / TILE;
    P.G = P.n_tiles < di->num_sms ? P.n_tiles : di->num_sms;
    if (P.G > MERGE_MAX_SPLITS) P.G = MERGE_MAX_SPLITS;
    P.scale = scale;
    P.out = static_cast<__half*>(out);
    P.err = di->err_word;
    void* ws;
    size_t ws_bytes;
    current_workspace(&ws, &ws_bytes);
    if (!ws || ws_bytes < paged_e4m3_workspace_bytes(R, ctx_len, di->num_sms))
        return GQA_ERR_WORKSPACE;
    float* w = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kWorkspaceCounterBytes);
    P.ws_o = w;
    P.ws_ml = w + (size_t)P.G * P.nq * D;
    CUtensorMap tk, tv;
    const uint64_t rows = (uint64_t)num_pages * PAGE;
    if (!make_map_2d_u8(&tk, kcache, rows, D, PAGE, 128) ||
        !make_map_2d_u8(&tv, vcache, rows, D, PAGE, 128))
        return GQA_ERR_CUDA;
    if (P.nq <= 16) return launch_np<16>(tk, tv, P, stream, di->device);
    if (P.nq <= 32) return launch_np<32>(tk, tv, P, stream, di->device);
    return launch_np<48>(tk, tv, P, stream, di->device);
}

}  // namespace gqa

// ---------------------------------------------------------------------------
// Allocation-free variant of the paged E4M3 tail.  It runs the same kernels
// but keeps the split partials in a file-scope device array instead of the
// caller-registered workspace, for callers that cannot allocate device memory.
#include <mutex>

namespace gqa {
namespace paged {

constexpr int kNoAllocMaxSplits = 160;
constexpr int kNoAllocMaxRows = 8 * HQ;  // query_rows <= 8
constexpr size_t kNoAllocFloats = (size_t)kNoAllocMaxSplits * kNoAllocMaxRows * (D + 2);

// Split partials (O, then (m, l)) of gqa_attn_paged_e4m3_noalloc: about
// 7.9 MB of module-scope device memory that every device loading the library
// holds until the process exits.  Host code must not use this name as a
// device pointer; the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) float g_noalloc_partials[kNoAllocFloats];

}  // namespace paged

size_t paged_e4m3_noalloc_capacity_floats() { return paged::kNoAllocFloats; }

int paged_e4m3_noalloc_launch(const void* q, const uint8_t* kcache, const uint8_t* vcache,
                              const float* kscale, const float* vscale,
                              const int32_t* block_table, int num_pages, int ctx_len, int R,
                              float scale, void* out, cudaStream_t stream) {
    using namespace paged;
    const DeviceInfo* di = device_info();
    if (!di) return GQA_ERR_CUDA;
    // Device address of the array, looked up once per device while that
    // device is current (the first call on a device does this).
    static float* s_addr[64] = {nullptr};
    static std::mutex s_mu;
    if (di->device >= 64) return GQA_ERR_CUDA;
    float* scratch;
    {
        std::lock_guard<std::mutex> lk(s_mu);
        if (!s_addr[di->device]) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_partials) != cudaSuccess || !p)
                return GQA_ERR_CUDA;
            s_addr[di->device] = static_cast<float*>(p);
        }
        scratch = s_addr[di->device];
    }
    Params P;
    P.kcache = kcache;
    P.vcache = vcache;
    P.kscale = kscale;
    P.vscale = vscale;
    P.table = block_table;
    P.q = static_cast<const __half*>(q);
    P.num_pages = num_pages;
    P.ctx_len = ctx_len;
    P.R = R;
    P.nq = R * HQ;
    P.n_tiles = (ctx_len + TILE - 1) / TILE;
    P.G = P.n_tiles < di->num_sms ? P.n_tiles : di->num_sms;
    if (P.G > kNoAllocMaxSplits) P.G = kNoAllocMaxSplits;
    P.scale = scale;
    P.out = static_cast<__half*>(out);
    P.err = di->err_word;
    if (P.nq > kNoAllocMaxRows || (size_t)P.G * P.nq * (D + 2) > kNoAllocFloats)
        return GQA_ERR_WORKSPACE;
    P.ws_o = scratch;
    P.ws_ml = scratch + (size_t)P.G * P.nq * D;
    CUtensorMap tk, tv;
    const uint64_t rows = (uint64_t)num_pages * PAGE;
    if (!make_map_2d_u8(&tk, kcache, rows, D, PAGE, 128) ||
        !make_map_2d_u8(&tv, vcache, rows, D, PAGE, 128))
        return GQA_ERR_CUDA;
    if (P.nq <= 16) return launch_np<16>(tk, tv, P, stream, di->device);
    if (P.nq <= 32) return launch_np<32>(tk, tv, P, stream, di->device);
    return launch_np<48>(tk, tv, P, stream, di->device);
}

}  // namespace gqa
