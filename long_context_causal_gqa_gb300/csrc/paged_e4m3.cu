// paged_e4m3.cu -- causal GQA verifier tail over an FP8-E4M3 paged KV cache.
//
// Problem ("[Perf] Ship the qualified SM70 long-context layout and drop its
// context fences", What / Changes): R <= 8 query rows (6R packed rows, Hq=6
// sharing Hkv=1) at the end of a context of up to 262144 keys; K and V are
// E4M3 bytes (one fp32 scale each) in page-16 blocks addressed through a
// block table of physical page ids; FP32 accumulation.  Here the page is any
// power of two in [8, 256], one launch may carry a batch of sequences with
// their context lengths read on the device, and other head groupings run one
// launch per KV head (R x Hq / Hkv <= 48 packed rows).  The page's operator
// decodes E4M3 through a shared lookup table and specialises the 8-row case;
// here the work is HBM-bound (one byte per K/V element) and shaped for sm_103a:
//
// * Split-KV: the context is cut into 128-key tiles (8 pages) and the tiles
//   into one contiguous range per SM.  Each split writes an (O, m, l) partial;
//   a merge kernel, launched as a programmatic dependent so that its launch
//   overlaps this kernel's tail, combines them (exact log-sum-exp merge).
// * Swap-AB UMMA on the FP8 tensor cores (kind::f8f6f4, K = 32 per
//   instruction): keys are the M=128 dimension, the packed query rows the N
//   dimension (NP = 16/32/48).  K and V enter as the raw E4M3 bytes the TMA
//   brought in, so nothing is decoded:
//     S^T[128 keys x 3NP] = K[128 x 256] . [Q1 | Q2 | Q3]^T        (K-major A)
//     O^T[128 d x 3NP]   += V^T[128 d x 128 keys] . [P1 | P2 | P3]^T
//                           (MN-major A, one UMMA chain per half of d)
//   Q and P are fp16 / fp32 quantities; each enters as a three-term E4M3
//   expansion x ~= t1 + t2 / 32 + t3 / 1024 (each term the E4M3 rounding of
//   the scaled remainder), which carries at least fp16's 11 significant bits,
//   so S = S1 + S2 / 32 + S3 / 1024 and likewise O.  Q uses one scale per
//   packed row (its absmax maps to 256); P <= 256 by the lazy rescale below.
//   With |x| <= 256 a remainder is at most half an E4M3 unit of x (<= 8), so
//   32 times it stays inside E4M3's range (448), and the smallest x the
//   expansion keeps is 2^-19 (E4M3's smallest subnormal, 2^-9, over 32^2).
//   K's and V's fp32 scales are applied to S and to the merged output.
// * Raw pages arrive by TMA tensor copies (128-byte swizzle, two 128-byte
//   halves of d per page) through a ring of 32 KB stages (K0, K1, V0, K2,
//   V1, ...: each V one tile behind its K, so that it arrives when its P is
//   ready); a stage is released by the commit of the UMMAs that read it.  The
//   ring is as deep as shared memory allows (6 stages for 16 packed rows):
//   under full load DRAM latency is several microseconds, and the bytes in
//   flight per SM set the bandwidth.  With
//   up to 32 packed rows S^T is double-buffered in tensor memory; at 48 the
//   three-term S^T and O^T leave room for one S^T buffer, which the softmax
//   releases as soon as it has read it.
// * Softmax over keys runs across TMEM lanes.  A per-row reference moves only
//   when a score exceeds it by more than 8 (log2 units, so P <= 256); it is
//   then set REF_SHIFT = 6 below the tile's exact max, so that right after a
//   move the largest P is 64 and the expansion's floor of 2^-19 sits at least
//   25 binades below the row's maximum (the fp16 P of the dense kernels
//   reaches 2^-24 below theirs).  The common case is one threshold compare and
//   a warpgroup vote per tile; the exact cross-lane max is taken only on the
//   first tile or when the vote fires.  Row sums stay per thread until the
//   split's end.
//
// Warp roles (64 + 128 NWG threads): 0 TMA producer, 1 TMEM owner + UMMA
// issuer, then NWG = 2 / 4 / 6 softmax warpgroups for 16 / 32 / 48 packed
// rows, each owning 8 of them (thread = TMEM lane = key).
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
namespace paged {

constexpr int D = kHeadDim;      // 256, the largest head size (sizes the static partials)
constexpr int TILE = 128;        // keys per tile
// Threads of a CTA with NWG softmax warpgroups: producer warp, UMMA warp,
// then 4 * NWG softmax warps.
__host__ __device__ constexpr int threads_for(int nwg) { return 64 + 128 * nwg; }
constexpr float RESCALE_THRESHOLD = 8.0f;

struct Params {
    const uint8_t* kcache;
    const uint8_t* vcache;
    const float* kscale;
    const float* vscale;
    const int32_t* table;
    const __half* q;
    const int* ctx_dev;   // device-side context lengths, one per sequence (nullptr: ctx_len)
    int batch;            // sequences sharing the grid (1 except for the batched entry point)
    int table_stride;     // block-table entries per sequence
    int page, log2_page;  // tokens per cache page, a power of two in [8, 256]
    int num_pages, ctx_len, R, nq, n_tiles, G;
    int hq;               // query heads per position in q / out
    FastDiv grp;          // packed rows per position in one launch (query heads of one KV head)
    float scale;
    int dh;         // head size, 256 or 128
    float* ws_o;    // [G][nq][dh] unnormalised partial O (in units of the E4M3 V)
    float* ws_ml;   // [G][nq][2]  (m in log2 units, l)
    __half* out;
    unsigned* err;
};

// Element offset of packed row r of sequence seq in q / out.  Packed row r is
// position r / grp of the sequence's tail and the (r mod grp)-th query head of
// the launch's KV head; q / out already point at that head group's first head.
__device__ __forceinline__ size_t row_offset(const Params& P, int seq, int r) {
    const int pos = P.grp.div(r);
    return ((size_t)(seq * P.R + pos) * P.hq + (r - pos * P.grp.d)) * P.dh;
}

// DH: head size, 256 or 128.  A K or V tile is TILE rows of DH E4M3 bytes:
// DH / 128 swizzle atoms ("halves") of 128 bytes per row.
template <int NP, int NWG, int DH>
struct Layout {
    static constexpr int HALVES = DH / 128;
    static constexpr int RAW_STAGE = TILE * DH;       // 32 KB (DH 256) or 16 KB per K or V tile
    static constexpr int NT = 3;                      // E4M3 expansion terms
    static constexpr int N3 = NT * NP;                // UMMA N
    // S^T buffers in tensor memory: two, except at 48 packed rows and DH 256,
    // where the three-term S^T and O^T leave room for one.
    static constexpr int NS = (NP <= 32 || DH == 128) ? 2 : 1;
    // P^T buffers: two, except at 48 rows and DH 256, where one buffer lets a
    // fifth raw stage fit (the copy stream's rate is set by its bytes in flight).
    static constexpr int NPT = (NP <= 32 || DH == 128) ? 2 : 1;
    // Raw K/V stages: 192 / 160 KB of 32 KB stages at DH 256; at DH 128 the
    // 16 KB stages come twice as many (the bytes in flight are what count).
    static constexpr int NRAW = DH == 256 ? ((NP <= 16) ? 6 : 5)
                                          : ((NP <= 16) ? 12 : (NP <= 32 ? 11 : 10));
    static constexpr int Q_BYTES = N3 * DH;           // [Q1|Q2|Q3]: N3 rows x DH B, in halves
    static constexpr int PT_BYTES = N3 * TILE;        // [P1|P2|P3]^T: N3 rows x 128 keys
    static constexpr int OFF_RAW = 0;
    static constexpr int OFF_Q = OFF_RAW + NRAW * RAW_STAGE;
    static constexpr int OFF_PT = OFF_Q + Q_BYTES;
    static constexpr int OFF_QS = OFF_PT + NPT * PT_BYTES;      // [NP] per-row Q scales
    static constexpr int OFF_RED = OFF_QS + NP * 4;             // [4 NWG warps][NP] floats
    static constexpr int OFF_MREF = OFF_RED + 4 * NWG * NP * 4;  // [NP] floats
    static constexpr int OFF_FAC = OFF_MREF + NP * 4;            // [NP] floats
    static constexpr int OFF_FLAG = OFF_FAC + NP * 4;            // [2][4 NWG] ints
    static constexpr int OFF_BAR = (OFF_FLAG + 2 * 4 * NWG * 4 + 7) & ~7;
    static constexpr int NUM_BARS = 40;   // >= NUM_BARRIERS
    static constexpr int OFF_TMEM = OFF_BAR + NUM_BARS * 8;
    static constexpr int BYTES = OFF_TMEM + 16;
    static constexpr int SMEM = BYTES + 1024;
    // TMEM columns
    static constexpr uint32_t S_COL = 0;              // NS buffers x N3  (S1 | S2 | S3)
    static constexpr uint32_t O_COL = NS * N3;        // HALVES x N3 (O1 | O2 | O3)
    static_assert(O_COL + HALVES * N3 <= 512, "tensor memory");
    static_assert(SMEM <= 232448, "shared memory");
    static_assert(NRAW <= 12, "raw stage barriers");
};

// mbarrier indices
constexpr int MAX_RAW = 12;
constexpr int MAX_WG = 6;
enum {
    B_RAW_FULL = 0,               // [MAX_RAW]
    B_RAW_EMPTY = MAX_RAW,        // [MAX_RAW]
    B_S_FULL = 2 * MAX_RAW,       // [2]
    B_P_READY = 2 * MAX_RAW + 2,  // [NPT]
    B_PT_EMPTY = 2 * MAX_RAW + 4, // [NPT] P.V of that P^T buffer done
    B_DRAIN = 2 * MAX_RAW + 6,
    B_GROUP = 2 * MAX_RAW + 7,    // [MAX_WG] per softmax warpgroup
    B_S_FREE = 2 * MAX_RAW + 7 + MAX_WG,  // single S^T buffer read by the softmax
    NUM_BARRIERS = B_S_FREE + 1,
};

static_assert(NUM_BARRIERS <= 40, "mbarrier slots");

// Copy order through the raw ring: K0, then K(j), V(j - 1) for j = 1 .. n - 1,
// then V(n - 1).  V(j) is requested one tile after K(j), so that it lands
// about when P(j) is ready instead of holding a stage while the softmax of
// tile j runs.
__device__ __forceinline__ int item_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int item_v(int j, int n) { return j == n - 1 ? 2 * n - 1 : 2 * j + 2; }

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

// Barrier among the 128 threads of one softmax warpgroup, built on an mbarrier
// so that it shares the bounded, abort-aware wait of the pipeline barriers: a
// thread that gave up elsewhere cannot leave the others blocked here forever.
__device__ __forceinline__ bool group_sync(uint32_t bar, uint32_t& phase, volatile int* abort,
                                           unsigned* err) {
    mbar_arrive(bar);
    const bool ok = mbar_wait(bar, phase, abort, err);
    phase ^= 1u;
    return ok;
}

// Which sequence, and which of its splits, CTA `split` works on.  With one
// sequence: all P.G splits.  With several (the batched tail): sequence b gets
// 1 + floor((G - batch) * tiles_b / total_tiles) splits, laid out in sequence
// order, from the context lengths read on the device; CTAs past the last
// sequence's splits get b = -1 and do nothing.  Device context lengths are
// clamped into [R, ctx_len] (bad = the value was outside).  Every warp runs
// this itself (lane-parallel over the sequences), so no block-wide step is
// needed before the CTA knows its work.
struct SplitOwner {
    int b, j, g, ctx;
    bool bad;
};
__device__ __forceinline__ int clamp_ctx(const Params& P, int c) {
    return c < P.R ? P.R : (c > P.ctx_len ? P.ctx_len : c);
}
__device__ __forceinline__ long long tiles_of(int ctx) { return (ctx + TILE - 1) / TILE; }

template <bool BATCHED>
__device__ SplitOwner split_owner(const Params& P, int split) {
    SplitOwner r;
    if (!BATCHED) {
        const int raw = P.ctx_dev ? *P.ctx_dev : P.ctx_len;
        r.b = 0;
        r.j = split;
        r.g = P.G;
        r.ctx = clamp_ctx(P, raw);
        r.bad = raw != r.ctx;
        return r;
    }
    const int lane = threadIdx.x & 31;
    long long total = 0;
    for (int i = lane; i < P.batch; i += 32) total += tiles_of(clamp_ctx(P, P.ctx_dev[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    const long long spare = P.G - P.batch;
    int base = 0;
    for (int i0 = 0; i0 < P.batch; i0 += 32) {
        const int i = i0 + lane;
        int ci = 0, gi = 0, bad = 0;
        if (i < P.batch) {
            const int raw = P.ctx_dev[i];
            ci = clamp_ctx(P, raw);
            bad = raw != ci;
            gi = 1 + (int)(spare * tiles_of(ci) / total);
        }
        int incl = gi;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        const int start = base + incl - gi;
        const unsigned m =
            __ballot_sync(0xffffffffu, i < P.batch && split >= start && split < start + gi);
        if (m) {
            const int src = __ffs(m) - 1;
            r.b = i0 + src;
            r.j = split - __shfl_sync(0xffffffffu, start, src);
            r.g = __shfl_sync(0xffffffffu, gi, src);
            r.ctx = __shfl_sync(0xffffffffu, ci, src);
            r.bad = __shfl_sync(0xffffffffu, bad, src) != 0;
            return r;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
    r.b = -1;
    r.j = r.g = r.ctx = 0;
    r.bad = false;
    return r;
}

// First split and split count of sequence b (the merge's view of split_owner).
__device__ void seq_splits(const Params& P, int b, int& first, int& count) {
    if (P.batch == 1) {
        first = 0;
        count = P.G;
        return;
    }
    const int lane = threadIdx.x & 31;
    long long total = 0;
    for (int i = lane; i < P.batch; i += 32) total += tiles_of(clamp_ctx(P, P.ctx_dev[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    const long long spare = P.G - P.batch;
    int base = 0;
    for (int i0 = 0; i0 <= b; i0 += 32) {
        const int i = i0 + lane;
        const int gi = i < P.batch ? 1 + (int)(spare * tiles_of(clamp_ctx(P, P.ctx_dev[i])) / total)
                                   : 0;
        int incl = gi;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        if (b < i0 + 32) {
            const int src = b - i0;
            first = base + __shfl_sync(0xffffffffu, incl - gi, src);
            count = __shfl_sync(0xffffffffu, gi, src);
            return;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
    first = count = 0;
}

template <int NP, int NWG, bool BATCHED, int DH>
__global__ void __launch_bounds__(threads_for(NWG), 1)
paged_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const Params P) {
    using L = Layout<NP, NWG, DH>;
    constexpr int HALVES = L::HALVES;
    constexpr int RAW_STAGE = L::RAW_STAGE;
    constexpr int NTHREADS = threads_for(NWG);
    constexpr int NKEY = 128 * NWG;   // softmax threads
    constexpr int NH = NP / NWG;      // packed query rows per softmax warpgroup
    static_assert(NP % NWG == 0 && NWG <= MAX_WG, "softmax split");
    constexpr int N3 = L::N3;    // UMMA N: three expansion terms
    constexpr int NS = L::NS;
    constexpr int NRAW = L::NRAW;
    constexpr int NPT = L::NPT;
    // E4M3 x E4M3 -> f32 (format fields 0 = E4M3 for kind::f8f6f4).
    constexpr uint32_t IDESC_QK = idesc_f16_f32(128, N3, false, false);
    constexpr uint32_t IDESC_PV = idesc_f16_f32(128, N3, true, false);   // A = V^T, MN-major

    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (sbase - smem_u32(smem_raw));
    const uint32_t s_raw = sbase + L::OFF_RAW;
    const uint32_t s_q = sbase + L::OFF_Q;
    const uint32_t s_pt = sbase + L::OFF_PT;
    float* qs = reinterpret_cast<float*>(gbase + L::OFF_QS);
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
    const int split = blockIdx.x;   // this CTA's partial slot
    // Launched as a programmatic dependent of the kernel before it on the
    // stream (the previous call's merge, in a model's consecutive layers): the
    // CTA launch overlaps that kernel, and nothing of global memory is read or
    // written before it has completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // Context length: the launch's, or read on the device (the grid is then
    // sized for the largest context, P.ctx_len, and splits past the actual
    // context get no tiles); with several sequences, this CTA's sequence.
    const SplitOwner own = split_owner<BATCHED>(P, split);
    if (own.b < 0) return;   // uniform: no sequence left for this CTA
    if (own.bad && own.j == 0 && threadIdx.x == 0) atomicOr(P.err, kErrBadCtxLen);
    const int ctx_len = own.ctx;
    const int n_tiles = (ctx_len + TILE - 1) / TILE;
    const int t_begin = (int)((long long)own.j * n_tiles / own.g);
    const int t_end = (int)((long long)(own.j + 1) * n_tiles / own.g);
    const int seq = own.b;
    const int ntl = t_end - t_begin;
    const int page = P.page, lpage = P.log2_page;
    const int n_logical = (ctx_len + page - 1) >> lpage;
    // The producer's first two chunks of block-table entries (one per lane),
    // requested before the barrier set-up so that their DRAM latency overlaps it.
    const int pg_begin = (t_begin * TILE) >> lpage;
    const int pg_end = ntl > 0 ? min(((t_end * TILE - 1) >> lpage) + 1, n_logical) : 0;
    const int32_t* table = P.table + (size_t)seq * P.table_stride;
    auto load_chunk = [&](int k) -> int {
        const int pg = pg_begin + 32 * k + lane;
        return pg < pg_end ? __ldg(table + pg) : 0;
    };
    int cur = 0, nxt = 0;
    if (warp == 0) {
        cur = load_chunk(0);
        nxt = load_chunk(1);
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < NRAW; ++s) {
            mbar_init(bar(B_RAW_FULL + s), 1);
            mbar_init(bar(B_RAW_EMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_S_FULL + b), 1);
            mbar_init(bar(B_P_READY + b), NKEY);
            mbar_init(bar(B_PT_EMPTY + b), 1);
        }
        for (int g = 0; g < NWG; ++g) mbar_init(bar(B_GROUP + g), 128);
        mbar_init(bar(B_S_FREE), NKEY);
        mbar_init(bar(B_DRAIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    // Barriers are initialised: the producer starts streaming at once, while
    // warps 1..9 build the Q operand and allocate tensor memory.
    __syncthreads();
    // The merge kernel may be scheduled now; it waits for this grid to finish.
    asm volatile("griddepcontrol.launch_dependents;");
    uint32_t tmem = 0;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // Block-table entries arrive a chunk of 32 pages (one per lane) ahead
        // of their use, so their latency stays off the copy stream.  A tile
        // covers TILE / page pages (page <= TILE, lane 2p + h copies page p,
        // half h of d) or a TILE-row slice of one page (page > TILE).
        if (ntl > 0) {
            const int ppt = page >= TILE ? 1 : TILE >> lpage;       // pages per tile, divides 32
            const int rows_per_copy = page >= TILE ? TILE : page;
            int cur_k = 0;
            // Lane HALVES * p + h copies page p, half h of d.
            const int pp = lane / HALVES, hh = lane % HALVES;
            uint32_t item = 0;
            bool ok = true;
            int id_prev = 0, npg_prev = 0, y_prev = 0;
            // One K or V stage: npg copies of rows_per_copy rows (row offset y0
            // inside the page when a tile is a slice of one page).
            auto issue = [&](const CUtensorMap* tm, int id, int npg, int y0) -> bool {
                const int s = item % NRAW;
                const uint32_t ph = (item / NRAW) & 1u;
                int okw = 1;
                if (lane == 0) {
                    okw = mbar_wait(bar(B_RAW_EMPTY + s), ph ^ 1u, abort_flag, P.err);
                    if (okw)
                        mbar_arrive_expect_tx(bar(B_RAW_FULL + s),
                                              (uint32_t)(npg * rows_per_copy * DH));
                }
                if (!__shfl_sync(0xffffffffu, okw, 0)) return false;
                // Stage layout: [2 halves of d][128 keys][128 B], 128B-swizzled.
                if (lane < HALVES * npg)
                    tma_load_2d(s_raw + s * RAW_STAGE + hh * (TILE * 128) +
                                    pp * (rows_per_copy * 128),
                                tm, bar(B_RAW_FULL + s), hh * 128, id * page + y0);
                ++item;
                return true;
            };
            for (int jj = 0; jj <= ntl && ok; ++jj) {
                int id = 0, npg = 0, y0 = 0;
                if (jj < ntl) {
                    const int tile = t_begin + jj;
                    const int lp0 = (tile * TILE) >> lpage;            // first logical page
                    const int rel = lp0 - pg_begin;
                    while ((rel >> 5) > cur_k) {
                        cur = nxt;
                        ++cur_k;
                        nxt = load_chunk(cur_k + 1);
                    }
                    npg = min(ppt, n_logical - lp0);
                    y0 = (tile * TILE) & (page - 1);
                    id = __shfl_sync(0xffffffffu, cur, (rel & 31) + (pp < ppt ? pp : 0));
                    if (lane < HALVES * npg && (id < 0 || id >= P.num_pages)) {
                        atomicOr(P.err, kErrBadPageId);
                        id = 0;
                    }
                    ok = issue(&tm_k, id, npg, y0);
                }
                if (ok && jj >= 1) ok = issue(&tm_v, id_prev, npg_prev, y_prev);
                id_prev = id;
                npg_prev = npg;
                y_prev = y0;
            }
            if (!ok && lane == 0) {
                for (int s = 0; s < NRAW; ++s) {
                    const uint32_t fills = item > (uint32_t)s ? (item - s + NRAW - 1) / NRAW : 0;
                    if (fills) drain_wait(bar(B_RAW_FULL + s), (fills - 1) & 1u);
                }
            }
        }
    } else {
        // ---- Q -> three-term E4M3 expansion [Q1 | Q2 | Q3] in shared memory
        // (K-major, 3NP rows of DH bytes in 128-byte halves, 128B-swizzled),
        // one scale per packed row: x / qs ~= t1 + t2 / 32 + t3 / 1024, |x / qs| <= 256.
        // Warps 1..9 take rows r = warp - 1, warp + 8, ...; all their loads are
        // issued before the first conversion.
        const float kscale = *P.kscale;
        {
            constexpr int QW = NTHREADS / 32 - 1;
            constexpr int RPW = (NP + QW - 1) / QW;
            constexpr int EPL = DH / 32;   // elements of a row per lane: 8 or 4
            using QV = typename std::conditional<EPL == 8, uint4, uint2>::type;
            const int d0 = lane * EPL;
            QV raw[RPW];
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                const int r = warp - 1 + QW * i;
                raw[i] = (r < P.nq) ? *reinterpret_cast<const QV*>(P.q + row_offset(P, seq, r) + d0)
                                    : QV{};
            }
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                const int r = warp - 1 + QW * i;
                if (r >= NP) break;
                float x[EPL];
                const __half* hx = reinterpret_cast<const __half*>(&raw[i]);
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
                uint8_t* qh = gbase + L::OFF_Q + h * (N3 * 128);
                if constexpr (EPL == 8) {
                    *reinterpret_cast<uint2*>(qh + sw128(r, cin >> 4) + (cin & 15)) =
                        make_uint2(w1[0], w1[1]);
                    *reinterpret_cast<uint2*>(qh + sw128(NP + r, cin >> 4) + (cin & 15)) =
                        make_uint2(w2[0], w2[1]);
                    *reinterpret_cast<uint2*>(qh + sw128(2 * NP + r, cin >> 4) + (cin & 15)) =
                        make_uint2(w3[0], w3[1]);
                } else {
                    *reinterpret_cast<uint32_t*>(qh + sw128(r, cin >> 4) + (cin & 15)) = w1[0];
                    *reinterpret_cast<uint32_t*>(qh + sw128(NP + r, cin >> 4) + (cin & 15)) = w2[0];
                    *reinterpret_cast<uint32_t*>(qh + sw128(2 * NP + r, cin >> 4) + (cin & 15)) =
                        w3[0];
                }
                if (lane == 0) qs[r] = sc;
            }
        }
        for (int c = threadIdx.x - 32; c < NP; c += NTHREADS - 32) mref[c] = -INFINITY;
        if (warp == 1) {
            tmem_alloc(smem_u32(tmem_ptr), 512);
            tmem_relinquish();
        }
        fence_async_shared();
        tc_fence_before();
        // Warps 1..9 only (the producer is already streaming); every one of them
        // reaches this barrier unconditionally.
        asm volatile("bar.sync 1, %0;" ::"r"(NTHREADS - 32) : "memory");
        tc_fence_after();
        tmem = *tmem_ptr;
        if (warp == 1) {
            // ------------------------------------------------------------ UMMA issuer
            if (lane == 0 && ntl > 0) {
                bool ok = true;
                auto stage_of = [](int item) { return item % NRAW; };
                auto phase_of = [](int item) { return (uint32_t)((item / NRAW) & 1); };
                auto issue_pv = [&](int x) -> bool {
                    if (!mbar_wait(bar(B_P_READY + x % NPT), (x / NPT) & 1, abort_flag, P.err))
                        return false;
                    const int vi = item_v(x, ntl);
                    if (!mbar_wait(bar(B_RAW_FULL + stage_of(vi)), phase_of(vi), abort_flag, P.err))
                        return false;
                    tc_fence_after();
                    const uint32_t vst = s_raw + stage_of(vi) * RAW_STAGE;
                    const uint32_t pt = s_pt + (x % NPT) * L::PT_BYTES;
#pragma unroll
                    for (int h = 0; h < HALVES; ++h) {
#pragma unroll
                        for (int ks = 0; ks < TILE / 32; ++ks) {
                            // V^T half h: M = 128 d (one 128-byte atom), K = 32 keys (rows)
                            const uint64_t a = sdesc_sw128(vst + h * (TILE * 128) + ks * 4096, 16384, 1024);
                            const uint64_t b = sdesc_sw128(pt + ks * 32, 16, 1024);
                            umma_f8(tmem + L::O_COL + h * N3, a, b, IDESC_PV, (x > 0 || ks > 0));
                        }
                    }
                    umma_commit(bar(B_PT_EMPTY + x % NPT));
                    umma_commit(bar(B_RAW_EMPTY + stage_of(vi)));
                    return true;
                };
                for (int jj = 0; jj < ntl && ok; ++jj) {
                    const int b = jj % NS;
                    const int ki = item_k(jj);
                    if (!mbar_wait(bar(B_RAW_FULL + stage_of(ki)), phase_of(ki), abort_flag, P.err)) {
                        ok = false;
                        break;
                    }
                    if (NS == 1 && jj > 0) {
                        // The single S^T buffer: the softmax must have read tile jj - 1.
                        if (!mbar_wait(bar(B_S_FREE), (uint32_t)((jj - 1) & 1), abort_flag, P.err)) {
                            ok = false;
                            break;
                        }
                    }
                    tc_fence_after();
                    const uint32_t kst = s_raw + stage_of(ki) * RAW_STAGE;
#pragma unroll
                    for (int kk = 0; kk < DH / 32; ++kk) {
                        const int h = kk >> 2;   // d half
                        const uint64_t a = sdesc_sw128(kst + h * (TILE * 128) + (kk & 3) * 32, 16, 1024);
                        const uint64_t bq = sdesc_sw128(s_q + h * (N3 * 128) + (kk & 3) * 32, 16, 1024);
                        umma_f8(tmem + L::S_COL + b * N3, a, bq, IDESC_QK, kk > 0);
                    }
                    umma_commit(bar(B_S_FULL + b));
                    umma_commit(bar(B_RAW_EMPTY + stage_of(ki)));
                    if (jj >= 1) ok = issue_pv(jj - 1);
                }
                if (ok) ok = issue_pv(ntl - 1);
                if (!ok) {
                    umma_commit(bar(B_DRAIN));
                    drain_wait(bar(B_DRAIN), 0);
                }
            }
        } else {
            // ------------------------------------------------------------ softmax warpgroups
            // Warpgroup hg owns packed query rows (S^T / O^T columns) hg*NH .. hg*NH+NH-1;
            // its lazy-rescale state is per column, so the two warpgroups never talk.
            const int hg = (warp - 2) >> 2;
            const int wq = warp & 3;
            const int wi = (warp - 2) & 3;                      // warp within the warpgroup
            const int k = wq * 32 + lane;                       // TMEM lane = key in tile = d in O^T half
            const int c0 = hg * NH;
            const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
            const int lim_base = ctx_len - P.R;                 // row r sees keys <= lim_base + r
            const uint32_t gbar = bar(B_GROUP + hg);
            uint32_t gphase = 0;
            // Score scale per packed row (log2 units): scale * kscale * Q row scale;
            // at 48 packed rows (72 registers per thread) read from shared memory
            // each tile (a broadcast) instead of held in registers.
            const float sl2k = P.scale * kscale * 1.4426950408889634f;
            constexpr bool kSl2InRegs = NP <= 32;
            float sl2[kSl2InRegs ? NH : 1];
#pragma unroll
            for (int c = 0; c < (kSl2InRegs ? NH : 1); ++c) sl2[c] = sl2k * qs[c0 + c];
            float lpart[NH];
#pragma unroll
            for (int c = 0; c < NH; ++c) lpart[c] = 0.f;
            // P^T store offsets: key k of row r = term * NP + c0 + c sits at byte
            // r * 128 + (((k >> 4) ^ (r & 7)) << 4) + (k & 15); c0 and NP are
            // multiples of 8, so r & 7 == c and the swizzled part depends only on
            // (k, c).
            static_assert(NH == 8 && NP % 8 == 0, "P^T store layout");
            const uint32_t p_row0 = (uint32_t)c0 * 128u + ((uint32_t)k & 15u);
            const uint32_t p_unit = ((uint32_t)k >> 4) << 4;
            auto pofs = [&](int c) -> uint32_t {
                return p_row0 + (uint32_t)c * 128u + (p_unit ^ ((uint32_t)c << 4));
            };
            bool ok = ntl > 0;
            for (int jj = 0; jj < ntl && ok; ++jj) {
                const int b = jj % NPT;          // P^T buffer
                const int sb = jj % NS;          // S^T buffer
                ok = mbar_wait(bar(B_S_FULL + sb), (uint32_t)((jj / NS) & 1), abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                float s[NH];
                {
                    uint32_t r1[NH], r2[NH], r3[NH];
                    tmem_ldn<NH>(t_lane + L::S_COL + sb * N3 + c0, r1);
                    tmem_ldn<NH>(t_lane + L::S_COL + sb * N3 + NP + c0, r2);
                    tmem_ldn<NH>(t_lane + L::S_COL + sb * N3 + 2 * NP + c0, r3);
                    tmem_ld_wait<NH>(r1);
                    tmem_ld_wait<NH>(r2);
                    tmem_ld_wait<NH>(r3);
                    if (NS == 1) {
                        // S^T is in registers: the next Q.K^T may overwrite it.
                        tc_fence_before();
                        mbar_arrive(bar(B_S_FREE));
                    }
#pragma unroll
                    for (int c = 0; c < NH; ++c)
                        s[c] = combine3(r1[c], r2[c], r3[c]) *
                               (kSl2InRegs ? sl2[kSl2InRegs ? c : 0] : sl2k * qs[c0 + c]);
                }
                const int key = (t_begin + jj) * TILE + k;
                if ((t_begin + jj) * TILE + TILE - 1 > lim_base) {
                    // Packed row cg (position cg / grp) sees the key iff
                    // cg / grp >= key - lim_base, i.e. cg >= (key - lim_base) grp.
                    const int need = (key - lim_base) * P.grp.d;
#pragma unroll
                    for (int c = 0; c < NH; ++c) {
                        const int cg = c0 + c;
                        const bool vis = (cg < P.nq) ? (cg >= need) : (key < ctx_len);
                        if (!vis) s[c] = -INFINITY;
                    }
                }
                // Vote: does any score exceed its row's reference max by > threshold?
                bool exceed = false;
#pragma unroll
                for (int c = 0; c < NH; ++c) exceed |= s[c] > mref[c0 + c] + RESCALE_THRESHOLD;
                const unsigned vote = __ballot_sync(0xffffffffu, exceed);
                volatile int* fl = flags + (jj & 1) * (4 * NWG) + hg * 4;
                if (lane == 0) fl[wi] = vote != 0;
                ok = group_sync(gbar, gphase, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                const bool any = fl[0] | fl[1] | fl[2] | fl[3];
                if (any) {
                    // Exact column max over the 128 keys of this tile.
#pragma unroll
                    for (int c = 0; c < NH; ++c) {
                        float m = s[c];
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                        if (lane == 0) red[(hg * 4 + wi) * NP + c0 + c] = m;
                    }
                    ok = group_sync(gbar, gphase, abort_flag, P.err);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    if (k < NH) {
                        const int c = c0 + k;
                        const float* rr = red + (hg * 4) * NP + c;
                        const float tmax = fmaxf(fmaxf(rr[0], rr[NP]), fmaxf(rr[2 * NP], rr[3 * NP]));
                        const float old = mref[c];
                        float f = 1.0f;
                        if (tmax > old + RESCALE_THRESHOLD) {
                            const float ref = tmax - REF_SHIFT;
                            f = (old == -INFINITY) ? 0.f : ex2(old - ref);
                            mref[c] = ref;
                        }
                        fac[c] = f;
                    }
                    ok = group_sync(gbar, gphase, abort_flag, P.err);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    if (jj > 0) {
                        // O^T must hold every earlier P.V before it is rescaled.
                        const int x = jj - 1;
                        ok = mbar_wait(bar(B_PT_EMPTY + x % NPT), (x / NPT) & 1, abort_flag, P.err);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                        tc_fence_after();
#pragma unroll
                        for (int g6 = 0; g6 < 3 * HALVES; ++g6) {   // (d half, expansion term)
                            const uint32_t col = L::O_COL + (g6 / 3) * N3 + (g6 % 3) * NP + c0;
                            uint32_t r[NH];
                            tmem_ldn<NH>(t_lane + col, r);
                            tmem_ld_wait<NH>(r);
#pragma unroll
                            for (int c = 0; c < NH; ++c)
                                r[c] = __float_as_uint(__uint_as_float(r[c]) * fac[c0 + c]);
                            tmem_stn<NH>(t_lane + col, r);
                        }
                        tmem_st_wait();
                    }
#pragma unroll
                    for (int c = 0; c < NH; ++c) lpart[c] *= fac[c0 + c];
                }
                // Keys past the context in the last tile (the rest of the last page,
                // or pages never loaded) hold whatever the cache or shared memory
                // held, possibly the E4M3 NaN code; zero their V rows so that
                // P = 0 times V stays 0.  Each warpgroup clears its share of the
                // row's 16-byte units (8 per half of d).
                if (t_begin + jj == n_tiles - 1 && (ctx_len & (TILE - 1)) != 0) {
                    const int vi = item_v(jj, ntl);
                    ok = mbar_wait(bar(B_RAW_FULL + vi % NRAW), (uint32_t)((vi / NRAW) & 1), abort_flag,
                                   P.err);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    if (key >= ctx_len) {
                        uint8_t* st = gbase + L::OFF_RAW + (vi % NRAW) * RAW_STAGE + k * 128;
                        for (int u = hg * 8 * HALVES / NWG; u < (hg + 1) * 8 * HALVES / NWG; ++u)
                            *reinterpret_cast<uint4*>(st + (u >> 3) * (TILE * 128) + (u & 7) * 16) =
                                make_uint4(0, 0, 0, 0);
                    }
                }
                // P^T buffer b is free once the P.V NPT tiles back has completed.
                ok = mbar_wait(bar(B_PT_EMPTY + b), ((jj / NPT) & 1) ^ 1, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                {
                    // [P1 | P2 | P3]^T, K-major: row = term * NP + packed row, byte = key.
                    uint8_t* pt = gbase + L::OFF_PT + b * L::PT_BYTES;
#pragma unroll
                    for (int c = 0; c < NH; c += 2) {
                        const float m0 = mref[c0 + c], m1 = mref[c0 + c + 1];
                        const float p0 = ex2(s[c] - (m0 == -INFINITY ? 0.f : m0));
                        const float p1 = ex2(s[c + 1] - (m1 == -INFINITY ? 0.f : m1));
                        lpart[c] += p0;
                        lpart[c + 1] += p1;
                        uint32_t t[3];
                        split3_e4m3x2(p0, p1, t[0], t[1], t[2]);
#pragma unroll
                        for (int e = 0; e < 3; ++e) {
                            pt[pofs(c) + e * NP * 128] = (uint8_t)(t[e] & 0xFF);
                            pt[pofs(c + 1) + e * NP * 128] = (uint8_t)(t[e] >> 8);
                        }
                    }
                }
                fence_async_shared();
                mbar_arrive(bar(B_P_READY + b));
            }
            // ---------------------------------------------------------- epilogue
            if (ok && ntl > 0) {
                const int x = ntl - 1;
                ok = mbar_wait(bar(B_PT_EMPTY + x % NPT), (x / NPT) & 1, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
            }
            if (ok && ntl > 0) {
                tc_fence_after();
                // Row sums: reduce the per-thread partial sums over the 128 keys.
#pragma unroll
                for (int c = 0; c < NH; ++c) {
                    float v = lpart[c];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == 0) red[(hg * 4 + wi) * NP + c0 + c] = v;
                }
                ok = group_sync(gbar, gphase, abort_flag, P.err);
                ok = __all_sync(0xffffffffu, ok);
            }
            if (ok && ntl > 0) {
                if (k < NH && c0 + k < P.nq) {
                    const int c = c0 + k;
                    const float* rr = red + (hg * 4) * NP + c;
                    const float l = (rr[0] + rr[NP]) + (rr[2 * NP] + rr[3 * NP]);
                    P.ws_ml[((size_t)split * P.nq + c) * 2 + 0] = mref[c];
                    P.ws_ml[((size_t)split * P.nq + c) * 2 + 1] = l;
                }
#pragma unroll
                for (int h = 0; h < HALVES; ++h) {
                    uint32_t r1[NH], r2[NH], r3[NH];
                    tmem_ldn<NH>(t_lane + L::O_COL + h * N3 + c0, r1);
                    tmem_ldn<NH>(t_lane + L::O_COL + h * N3 + NP + c0, r2);
                    tmem_ldn<NH>(t_lane + L::O_COL + h * N3 + 2 * NP + c0, r3);
                    tmem_ld_wait<NH>(r1);
                    tmem_ld_wait<NH>(r2);
                    tmem_ld_wait<NH>(r3);
                    const int d = h * 128 + k;
#pragma unroll
                    for (int c = 0; c < NH; ++c)
                        if (c0 + c < P.nq)
                            P.ws_o[((size_t)split * P.nq + c0 + c) * DH + d] =
                                combine3(r1[c], r2[c], r3[c]);
                }
            }
            if (ntl == 0 && k < NH && c0 + k < P.nq) {
                // A split with no tiles (a device-side context shorter than the
                // one the grid was sized for): a partial the merge gives zero
                // weight; its O is never read.
                P.ws_ml[((size_t)split * P.nq + c0 + k) * 2 + 0] = -INFINITY;
                P.ws_ml[((size_t)split * P.nq + c0 + k) * 2 + 1] = 0.f;
            }
        }

    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// out[c, d] = vscale * sum_s w_s O_s[c, d] / sum_s w_s l_s, w_s = 2^(m_s - M).
// Block (c, dh) merges packed row c for d = 128 dh .. 128 dh + 127, four d per
// lane.  Warp w owns the splits s = w, w + 16, ...; the first MERGE_PF of them
// are loaded together with every split's (m, l), so that one round of L2
// latency covers up to 16 * MERGE_PF splits.  The warp sums are added in warp order,
// so the result does not depend on timing.  The kernel is launched as a
// programmatic dependent of the split kernel: everything before
// griddepcontrol.wait overlaps the split kernel's last CTAs.
constexpr int MERGE_MAX_SPLITS = 1024;
constexpr int MERGE_WARPS = 16;
constexpr int MERGE_PF = 10;

__global__ void __launch_bounds__(MERGE_WARPS * 32) paged_merge_kernel(const Params P) {
    __shared__ float w_s[MERGE_MAX_SPLITS];
    __shared__ float4 red[MERGE_WARPS][32];
    __shared__ float wred[2][MERGE_WARPS];
    const int seq = P.batch > 1 ? (int)blockIdx.x / P.nq : 0;   // sequence
    const int c = (int)blockIdx.x - seq * P.nq;                   // packed row within it
    const size_t out_off = row_offset(P, seq, c);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int d0 = blockIdx.y * 128 + lane * 4;
    // The next call's split kernel may launch now (it occupies no SM this
    // kernel needs until these blocks are resident, and reads nothing before
    // this grid has completed).
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    int S0 = 0, G = P.G;                    // this sequence's splits S0 .. S0 + G - 1
    if (P.batch > 1) seq_splits(P, seq, S0, G);
    const float vs = *P.vscale;
    // One round of loads: the O partials of this warp's first MERGE_PF splits
    // and the (m, l) pairs of the splits threadIdx.x + 512 i.
    float4 o[MERGE_PF];
#pragma unroll
    for (int i = 0; i < MERGE_PF; ++i) {
        const int s = warp + MERGE_WARPS * i;
        o[i] = s < G ? __ldcg(reinterpret_cast<const float4*>(P.ws_o + ((size_t)(S0 + s) * P.nq + c) * P.dh + d0))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    constexpr int ML_PT = MERGE_MAX_SPLITS / (MERGE_WARPS * 32);
    float2 ml[ML_PT];
#pragma unroll
    for (int i = 0; i < ML_PT; ++i) {
        const int s = threadIdx.x + MERGE_WARPS * 32 * i;
        ml[i] = s < G ? __ldcg(reinterpret_cast<const float2*>(P.ws_ml + ((size_t)(S0 + s) * P.nq + c) * 2))
                      : make_float2(-INFINITY, 0.f);
    }
    // M = max_s m_s.
    float mx = ml[0].x;
#pragma unroll
    for (int i = 1; i < ML_PT; ++i) mx = fmaxf(mx, ml[i].x);
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
    if (lane == 0) wred[0][warp] = mx;
    __syncthreads();
    float M = wred[0][0];
#pragma unroll
    for (int w = 1; w < MERGE_WARPS; ++w) M = fmaxf(M, wred[0][w]);
    // w_s = 2^(m_s - M), L = sum_s w_s l_s.
    float lsum = 0.f;
#pragma unroll
    for (int i = 0; i < ML_PT; ++i) {
        const int s = threadIdx.x + MERGE_WARPS * 32 * i;
        const float w = (ml[i].x == -INFINITY) ? 0.f : exp2f(ml[i].x - M);
        if (s < G) w_s[s] = w;
        lsum += w * ml[i].y;
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o2);
    if (lane == 0) wred[1][warp] = lsum;
    __syncthreads();
    // A zero weight (a split that saw no visible key, or none at all) skips
    // its O, which may hold anything.
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [&](float w, const float4& v) {
        if (w != 0.f) {
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
    };
#pragma unroll
    for (int i = 0; i < MERGE_PF; ++i) {
        const int s = warp + MERGE_WARPS * i;
        add(s < G ? w_s[s] : 0.f, o[i]);
    }
    for (int s = warp + MERGE_WARPS * MERGE_PF; s < G; s += MERGE_WARPS) {
        const float w = w_s[s];
        if (w != 0.f)
            add(w, __ldcg(reinterpret_cast<const float4*>(P.ws_o + ((size_t)(S0 + s) * P.nq + c) * P.dh + d0)));
    }
    red[warp][lane] = acc;
    __syncthreads();
    if (warp == 0) {
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < MERGE_WARPS; ++w) L += wred[1][w];
        float4 a = red[0][lane];
#pragma unroll
        for (int w = 1; w < MERGE_WARPS; ++w) {
            const float4 b = red[w][lane];
            a.x += b.x;
            a.y += b.y;
            a.z += b.z;
            a.w += b.w;
        }
        const float f = L > 0.f ? vs / L : 0.f;
        const __half2 h01 = __floats2half2_rn(a.x * f, a.y * f);
        const __half2 h23 = __floats2half2_rn(a.z * f, a.w * f);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t*>(&h01);
        pk.y = *reinterpret_cast<const uint32_t*>(&h23);
        *reinterpret_cast<uint2*>(P.out + out_off + d0) = pk;
    }
}

template <int NP, int NWG, bool BATCHED, int DH>
int launch_np_b(const CUtensorMap& tk, const CUtensorMap& tv, Params& P, cudaStream_t stream,
                int device) {
    using L = Layout<NP, NWG, DH>;
    (void)device;
    if (ensure_smem_limit(reinterpret_cast<const void*>(paged_split_kernel<NP, NWG, BATCHED, DH>),
                          L::SMEM) != GQA_OK)
        return GQA_ERR_CUDA;
    // Both kernels are programmatic dependents of the kernel before them.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(P.G);
    cfg.blockDim = dim3(threads_for(NWG));
    cfg.dynamicSmemBytes = L::SMEM;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, paged_split_kernel<NP, NWG, BATCHED, DH>, tk, tv, P) !=
        cudaSuccess)
        return GQA_ERR_CUDA;
    cfg.gridDim = dim3(P.batch * P.nq, P.dh / 128);
    cfg.blockDim = dim3(MERGE_WARPS * 32);
    cfg.dynamicSmemBytes = 0;
    if (cudaLaunchKernelEx(&cfg, paged_merge_kernel, P) != cudaSuccess) return GQA_ERR_CUDA;
    return GQA_OK;
}

// Packed query rows -> UMMA N and softmax warpgroups: every softmax thread
// owns 8 columns (8-aligned in tensor memory), so that the latency-bound
// softmax chain is spread over 8, 16 or 24 warps.
template <int NP, int NWG, int DH>
int launch_np(const CUtensorMap& tk, const CUtensorMap& tv, Params& P, cudaStream_t stream,
              int device) {
    // One sequence (the common tail) or several (the batched entry point):
    // separate instantiations, so the single-sequence kernel carries none of
    // the batched bookkeeping.
    return P.batch > 1 ? launch_np_b<NP, NWG, true, DH>(tk, tv, P, stream, device)
                       : launch_np_b<NP, NWG, false, DH>(tk, tv, P, stream, device);
}

template <int DH>
int launch_split_dh(const CUtensorMap& tk, const CUtensorMap& tv, Params& P,
                    cudaStream_t stream, int device) {
    if (P.nq <= 16) return launch_np<16, 2, DH>(tk, tv, P, stream, device);
    if (P.nq <= 32) return launch_np<32, 4, DH>(tk, tv, P, stream, device);
    return launch_np<48, 6, DH>(tk, tv, P, stream, device);
}

int launch_split(const CUtensorMap& tk, const CUtensorMap& tv, Params& P, cudaStream_t stream,
                 int device) {
    return P.dh == 128 ? launch_split_dh<128>(tk, tv, P, stream, device)
                       : launch_split_dh<256>(tk, tv, P, stream, device);
}

// Grouping fields: Hq query heads per position, Hkv KV heads, each shared by
// Hq / Hkv query heads; one launch takes one KV head's R * Hq / Hkv packed rows.
void set_grouping(Params& P, int Hq, int Hkv) {
    P.hq = Hq;
    P.grp = make_fastdiv(Hq / Hkv);
    P.nq = P.R * (Hq / Hkv);
}

// Split + merge once per KV head.  Head g reads row g of every cache token
// (the caches [num_pages * page, Hkv, dh] seen as rows Hkv * dh bytes apart) and
// writes query heads g * grp .. g * grp + grp - 1.  Launches on one stream run
// in order, so they can share the split partials.
int launch_heads(Params& P, const void* q, void* out, const uint8_t* kcache,
                 const uint8_t* vcache, int Hkv, cudaStream_t stream, int device) {
    const uint64_t rows = (uint64_t)P.num_pages * P.page;
    const uint32_t box_rows = P.page < TILE ? (uint32_t)P.page : (uint32_t)TILE;
    const int dh = P.dh;
    for (int g = 0; g < Hkv; ++g) {
        CUtensorMap tk, tv;
        if (!make_map_2d_u8(&tk, kcache + (size_t)g * dh, rows, dh, (uint64_t)Hkv * dh, box_rows,
                            128) ||
            !make_map_2d_u8(&tv, vcache + (size_t)g * dh, rows, dh, (uint64_t)Hkv * dh, box_rows,
                            128))
            return GQA_ERR_CUDA;
        P.q = static_cast<const __half*>(q) + (size_t)g * P.grp.d * dh;
        P.out = static_cast<__half*>(out) + (size_t)g * P.grp.d * dh;
        const int rc = launch_split(tk, tv, P, stream, device);
        if (rc != GQA_OK) return rc;
    }
    return GQA_OK;
}

}  // namespace paged

size_t paged_e4m3_workspace_bytes(int nq, int ctx_len, int num_sms, int Dh) {
    const int n_tiles = (ctx_len + paged::TILE - 1) / paged::TILE;
    const int G = n_tiles < num_sms ? n_tiles : num_sms;
    return kWorkspaceCounterBytes + (size_t)G * nq * (Dh + 2) * sizeof(float) + 256;
}

int paged_e4m3_launch(const void* q, const uint8_t* kcache, const uint8_t* vcache,
                      const float* kscale, const float* vscale, const int32_t* block_table,
                      int num_pages, int page, int ctx_len, const int* ctx_dev, int R,
                      int Hq, int Hkv, int Dh, float scale, void* out, cudaStream_t stream) {
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
    P.ctx_dev = ctx_dev;
    P.batch = 1;
    P.table_stride = 0;
    P.page = page;
    P.log2_page = __builtin_ctz((unsigned)page);
    P.num_pages = num_pages;
    P.ctx_len = ctx_len;
    P.R = R;
    P.dh = Dh;
    set_grouping(P, Hq, Hkv);
    P.n_tiles = (ctx_len + TILE - 1) / TILE;
    P.G = P.n_tiles < di->num_sms ? P.n_tiles : di->num_sms;
    if (P.G > MERGE_MAX_SPLITS) P.G = MERGE_MAX_SPLITS;
    P.scale = scale;
    P.out = static_cast<__half*>(out);
    P.err = di->err_word;
    void* ws;
    size_t ws_bytes;
    current_workspace(&ws, &ws_bytes);
    if (!ws || ws_bytes < paged_e4m3_workspace_bytes(P.nq, ctx_len, di->num_sms, Dh))
        return GQA_ERR_WORKSPACE;
    float* w = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kWorkspaceCounterBytes);
    P.ws_o = w;
    P.ws_ml = w + (size_t)P.G * P.nq * Dh;
    return launch_heads(P, q, out, kcache, vcache, Hkv, stream, di->device);
}

size_t paged_e4m3_batch_workspace_bytes(int nq, int batch, int num_sms, int Dh) {
    const int G = batch > num_sms ? batch : num_sms;
    return kWorkspaceCounterBytes + (size_t)G * nq * (Dh + 2) * sizeof(float) + 256;
}

// Several sequences' tails in one launch: q/out [batch, R, Hq, 256], block
// tables [batch, table_stride], context lengths read on the device.  The grid
// has max(SMs, batch) splits, shared out between the sequences in proportion
// to their tile counts (split_owner).
int paged_e4m3_batch_launch(const void* q, const uint8_t* kcache, const uint8_t* vcache,
                            const float* kscale, const float* vscale,
                            const int32_t* block_tables, int table_stride, int num_pages,
                            int page, const int* ctx_lens_dev, int max_ctx_len, int batch,
                            int R, int Hq, int Hkv, int Dh, float scale, void* out,
                            cudaStream_t stream) {
    using namespace paged;
    const DeviceInfo* di = device_info();
    if (!di) return GQA_ERR_CUDA;
    Params P;
    P.kcache = kcache;
    P.vcache = vcache;
    P.kscale = kscale;
    P.vscale = vscale;
    P.table = block_tables;
    P.q = static_cast<const __half*>(q);
    P.ctx_dev = ctx_lens_dev;
    P.batch = batch;
    P.table_stride = table_stride;
    P.page = page;
    P.log2_page = __builtin_ctz((unsigned)page);
    P.num_pages = num_pages;
    P.ctx_len = max_ctx_len;
    P.R = R;
    P.dh = Dh;
    set_grouping(P, Hq, Hkv);
    P.n_tiles = (max_ctx_len + TILE - 1) / TILE;
    P.G = batch > di->num_sms ? batch : di->num_sms;
    if (P.G > MERGE_MAX_SPLITS) return GQA_ERR_UNSUPPORTED;
    P.scale = scale;
    P.out = static_cast<__half*>(out);
    P.err = di->err_word;
    void* ws;
    size_t ws_bytes;
    current_workspace(&ws, &ws_bytes);
    if (!ws || ws_bytes < paged_e4m3_batch_workspace_bytes(P.nq, batch, di->num_sms, Dh))
        return GQA_ERR_WORKSPACE;
    float* w = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kWorkspaceCounterBytes);
    P.ws_o = w;
    P.ws_ml = w + (size_t)P.G * P.nq * Dh;
    return launch_heads(P, q, out, kcache, vcache, Hkv, stream, di->device);
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
constexpr int kNoAllocMaxRows = 48;  // packed rows per launch
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
                              const int32_t* block_table, int num_pages, int page, int ctx_len,
                              int R, int Hq, int Hkv, int Dh, float scale, void* out,
                              cudaStream_t stream) {
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
    P.ctx_dev = nullptr;
    P.batch = 1;
    P.table_stride = 0;
    P.page = page;
    P.log2_page = __builtin_ctz((unsigned)page);
    P.num_pages = num_pages;
    P.ctx_len = ctx_len;
    P.R = R;
    P.dh = Dh;
    set_grouping(P, Hq, Hkv);
    P.n_tiles = (ctx_len + TILE - 1) / TILE;
    P.G = P.n_tiles < di->num_sms ? P.n_tiles : di->num_sms;
    if (P.G > kNoAllocMaxSplits) P.G = kNoAllocMaxSplits;
    P.scale = scale;
    P.out = static_cast<__half*>(out);
    P.err = di->err_word;
    if (P.nq > kNoAllocMaxRows || (size_t)P.G * P.nq * (Dh + 2) > kNoAllocFloats)
        return GQA_ERR_WORKSPACE;
    P.ws_o = scratch;
    P.ws_ml = scratch + (size_t)P.G * P.nq * Dh;
    return launch_heads(P, q, out, kcache, vcache, Hkv, stream, di->device);
}

}  // namespace gqa
