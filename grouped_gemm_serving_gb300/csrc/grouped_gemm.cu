// moe_grouped_gemm: the per-expert GEMMs of the MoE layer on the
// fifth-generation tensor cores (tcgen05.mma, accumulators in tensor memory),
// operands staged by TMA.
//
// Sources: group_gemm_same_nk for fc1 and fc2 with silu(gate) * up between
// them (section 1 of "LlamaFactory Triton fused MoE kernel");
// grouped_fp8_matmul with 128x128-block weight scales and per-token,
// per-128-column activation scales (section 1 of "Hugging Face Transformers:
// MoE and FP8 kernel optimisation"); sentinel rows neither computed nor left
// uninitialised (sections 2 and 3 of the same write-up); one grouped GEMM
// over rows sorted by expert id (grouped_mm backend, "Mixture of Experts in
// transformers").
//
// Two kernels share the code below (one persistent CTA per SM, 384 threads).
//
// bf16 (SWAP): swapped operands on CTA pairs (clusters of two, tcgen05
// cta_group::2).  A pair tile is 256 weight rows (128 per CTA) x the tokens of
// one token tile of one expert (up to 256, split equally within the expert,
// the MMA's N rounded up to 16), so the tokens of an expert pad to a multiple
// of 16 instead of 128.  Each CTA stages its 128 weight rows and half the
// token rows (up to 32 KB per k-block, seven deep);
// the even CTA issues the MMAs for both and commits to both CTAs' barriers;
// each CTA's accumulator holds its weight rows x all tokens of the tile.
// SwiGLU: a CTA's 128 weight rows are its 64 features' gate and up rows,
// interleaved in groups of 8 (8 gate rows, the same 8 up rows, ...), so a
// feature's gate and up accumulators sit 8 lanes apart in one warp: the two
// lanes swap half of each 32-token chunk with one shuffle per token and
// both compute silu(g) * u.  An expert's last SwiGLU tile, when at most 64 of
// its 128 features exist (I = 2880: 2880 = 22.5 x 128), is an M = 128 pair
// MMA instead (N rounded up to 32): each CTA stages 64 weight rows (32
// features) and its accumulator holds weight row l % 64 for tokens
// (l / 64) * N/2 + column in lane l, columns below N/2.  So is an expert's
// last store tile with at most 128 of its 256 features (forward and data
// gradient; the weight gradient keeps M = 256 there, which measured faster).
//
// FP8 (and gathered A): single CTAs, 128 rows (tokens) x 256 columns
// (weights), 48 KB per k-block, four deep.  Each 128-wide k-block is an exact
// e4m3 x e4m3 partial in TMEM; the epilogue promotes it with
// sa[row, kb] * sb[block, kb] into fp32 registers while the MMA fills the
// other buffer.
//
// Roles:
//   warp 0      TMA producer
//   warp 1      MMA issuer (in a pair, the even CTA's only)
//   warps 2-3   idle (they complete warpgroup 0 for the FP8 register split),
//               except with gathered A (below)
//   warps 4-11  epilogue: tcgen05.ld the accumulator, apply the epilogue and
//               store; warp w reads TMEM lanes 32*(w%4).., columns half
//               (w-4)/4; then zero the sentinel rows [offsets[E], M_cap).
// The producer and MMA loops run on the whole warp and let one elected lane
// issue: TMA and tcgen05 instructions take warp-uniform operands, and issued
// from a single-thread branch they cost several times as many cycles.
// Accumulators are double-buffered across tiles in TMEM (2 x 256 columns).
// The tile list is built on the device from offsets, ordered expert-major,
// then weight tile, then token tile, so CTAs that run at the same time share
// a weight tile in L2.  No tile is issued for sentinel rows.
//
// Gathered A (moe_grouped_gemm_gather): instead of one tile load from a
// permuted buffer, the A tile is fetched four rows at a time with TMA
// tile::gather4 loads straight from token order (row p = x[sorted_rows[p] /
// k]), into the same 128-byte-swizzled layout and counted on the same stage
// barrier as the weight tile; only the quads that hold live rows are fetched.
// The gathers of a stage are shared by warps 0, 2 and 3 (one issuing lane
// each).  This folds the scatter of "LlamaFactory Triton fused MoE kernel"
// (section 1) into the first GEMM.  A gather4 costs far more than a quarter of
// a 128-row tile load, and every A tile is fetched again for each column tile,
// so with full tiles the separate scatter is faster.
//
// Every mbarrier wait is bounded (2 s): on expiry the CTA records
// MOE_DEVERR_TIMEOUT, stops all roles, waits (bounded) for its in-flight TMA
// loads and MMAs, frees its tensor memory and exits.
#include <cuda_fp8.h>
#include <cudaTypedefs.h>

#include <climits>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = 128 + kEpiThreads;  // warpgroup 0: TMA, MMA, 2 idle warps
constexpr uint32_t kTmemCols = 2 * BN;
constexpr int kStageA = BM * 128;
constexpr int kStageB = BN * 128;
enum Epi { EPI_STORE = 0, EPI_SWIGLU = 1, EPI_SWIGLU_Q = 2 };

// Stage ring: a single-CTA tile stages 128 A + 256 B rows (48 KB) four deep;
// a CTA of a pair stages up to 128 + 128 rows (32 KB) seven deep: its
// epilogues need no shared memory beyond the ring and the barriers (pair
// kernels allocate no Aux block, see smem_bytes).
constexpr int kMaxStages = 7;
template <bool PAIR, int EPI>
struct Geo {
    static constexpr int kStages = PAIR ? 7 : 4;
    static constexpr int kStageBytes = PAIR ? kStageA + kStageB / 2 : kStageA + kStageB;
};
constexpr int kMaxE = 256;
constexpr int kScaleRing = 4;   // k-blocks of block-scale prefetch in the FP8 epilogue
constexpr int kGatherWarps = 3; // warps 0, 2, 3 issue the row gathers of gathered A
// Swapped operands on CTA pairs (bf16): the weights are the M = 256 rows of
// a tcgen05 cta_group::2 MMA (128 per CTA) and an expert's tokens its N = up
// to BT columns (N/2 rows in each CTA's shared memory), so a tile pads the
// expert's rows to a multiple of 16 instead of 128, and each SM loads up to 32 KB
// of operands per k-block instead of 48 KB.
constexpr int BT = 256;
constexpr int kSwapFeatSwiglu = 128;  // h features per pair tile (each CTA: 64 gate + 64 up rows)
constexpr int kSwapFeatStore = 256;   // output features per pair tile (128 per CTA)
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kDrainNs = 100000000ull;
constexpr int kRegsLow = 56, kRegsHigh = 224;
static_assert(128 * kRegsLow + kEpiThreads * kRegsHigh <= kThreads * 168,
              "register split exceeds the launch allocation");
static_assert(kGatherWarps >= 1 && kGatherWarps <= 3, "gathering warps are 0, 2 and 3 of warpgroup 0");

struct Params {
    const int32_t* offsets;
    const float* a_scales;  // FP8: [K/128, M_cap]; gathered: [T, K/128]
    const float* b_scales;  // FP8: [E, nb_scale, K/128]
    void* out;              // bf16 [M_cap, out_cols], or e4m3 for EPI_SWIGLU_Q
    float* out_scales;      // EPI_SWIGLU_Q: [out_cols/128, M_cap]
    int* err;
    int E, M_cap, N, K;
    int half;      // SwiGLU: N/2 (gate rows [0, half), up rows [half, N))
    int out_cols;  // N (store) or N/2 (SwiGLU)
    int n_tiles, k_blocks, nb_scale;
    // gathered A (gx != nullptr): row p of A is row sorted_rows[p] / topk of gx
    const uint8_t* gx;
    const int32_t* sorted_rows;
    int T, topk;
    // weight-gradient kernel (WG: pair, bf16 store): the "weights" are A
    // [M_cap, out_cols] and the "tokens" dC [M_cap, wg_rows], both read
    // MN-major over the expert's own rows; every expert has all
    // wg_rows x out_cols output tiles over its own k-blocks; the output is
    // [E, wg_rows, out_cols].
    int wg_rows;
    // swapped store tiles only: the weights are MN-major, B [E, K, N] with
    // the N output features contiguous (the data gradient reads the forward
    // weights [E, N_fwd, K_fwd] in place this way)
    int mn_a;
    // swapped store tiles only: the weighted combine fused into the epilogue
    // (moe_grouped_gemm_combine).  sorted_rows and topk (above) map a row to
    // its token; counters [T, nfb] count the stored slots of each (token,
    // 128-feature block) and start at zero.
    int fc;
    const int32_t* ids;
    const float* wts;
    const int32_t* row_pos;
    int* counters;
    int nfb;
    void* cout;   // out bf16 [T, out_cols]
};

// Shared memory after the stage ring: barriers and the tile list (every
// mode), then the Aux block of the modes that need it.
struct alignas(16) Shared {
    uint64_t full[kMaxStages], empty[kMaxStages];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t xbar[2];  // amax exchange of the quantising epilogue
    uint64_t mma_done;
    uint64_t cbar;     // fused combine: every epilogue thread has stored its rows of the tile
    uint32_t tmem_base;
    int abort_flag;
    int valid;
    int prefix[kMaxE + 1];  // exclusive prefix over experts of row-tile counts
};
struct alignas(16) Aux {
    alignas(16) int gtok[kGatherWarps][BM];  // gathered A: each issuing warp's copy of the tile's tokens
    float amax_x[2][2][BM];  // quantising epilogue
    float scale_ring[kScaleRing * 3 * kEpiThreads];  // FP8 block scales in flight
};
// The Aux block sits right after Shared; the single-CTA kernels allocate it,
// and only their code paths reach it.
__device__ __forceinline__ Aux& aux(Shared& S) {
    return *reinterpret_cast<Aux*>(reinterpret_cast<uint8_t*>(&S) + sizeof(Shared));
}

template <bool PAIR, int EPI>
constexpr size_t smem_bytes() {
    using G = Geo<PAIR, EPI>;
    constexpr bool with_aux = !PAIR;
    return 1024 + static_cast<size_t>(G::kStages) * G::kStageBytes + sizeof(Shared) + (with_aux ? sizeof(Aux) : 0);
}
static_assert(smem_bytes<false, EPI_STORE>() <= 227 * 1024 && smem_bytes<false, EPI_SWIGLU_Q>() <= 227 * 1024 &&
                  smem_bytes<true, EPI_STORE>() <= 227 * 1024 && smem_bytes<true, EPI_SWIGLU>() <= 227 * 1024,
              "shared memory per CTA");

// Tensor maps over the token operand of the swapped kernels with boxes of
// 8, 16, .., 128 rows: a CTA's half of a token tile is one box of exactly
// its height.
// The weight gradient puts its four operand maps in the first slots instead:
// A and dC in place, then their zero-padded tails (64 features x 64 rows
// boxes, MN-major).
constexpr int kTokenMaps = 16;
struct TokenMaps {
    CUtensorMap m[kTokenMaps];
};
constexpr int kWgA = 0, kWgC = 1, kWgTailA = 2, kWgTailC = 3, kWgMaps = 4;

struct Tile {
    int e, row0, row_end, col0;
    int rows;  // swapped: token rows of this tile (<= BT)
    // swapped forward and data gradient: the expert's last feature tile, at
    // most half used (<= 64 h features for SwiGLU, <= 128 features for a
    // store), runs as an M = 128 pair MMA (64 weight rows per CTA)
    bool half;
    int nkb;    // the tile's k-blocks
    int first;  // weight gradient: the expert's first row
};

// Weight gradient: every expert has the same wg_pair_mt(p) token tiles.
__device__ __forceinline__ int wg_pair_mt(const Params& p) { return (p.wg_rows + BT - 1) / BT; }

template <bool SWAP, bool WG = false>
__device__ __forceinline__ Tile decode_tile(int t, const Shared& S, const Params& p) {
    static_assert(!WG || SWAP, "the weight gradient runs on CTA pairs");
    int lo = 0, mt, local;
    if (WG) {
        // every expert has mt x n_tiles tiles; S.prefix is its k-block prefix
        mt = wg_pair_mt(p);
        lo = t / (mt * p.n_tiles);
        local = t - lo * mt * p.n_tiles;
    } else {
        int hi = p.E;  // largest e < E with prefix[e] * n_tiles <= t
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (S.prefix[mid] * p.n_tiles <= t) lo = mid; else hi = mid;
        }
        mt = S.prefix[lo + 1] - S.prefix[lo];
        local = t - S.prefix[lo] * p.n_tiles;
    }
    Tile ti;
    ti.e = lo;
    ti.row_end = p.offsets[lo + 1];
    ti.first = 0;
    ti.nkb = p.k_blocks;
    ti.half = false;
    if (WG) {
        // weight gradient on a pair: the tokens are the wg_rows output rows
        // in tiles of BT; the contraction runs over the expert's own rows in
        // k-blocks of 64 (S.prefix is the k-block prefix)
        ti.row0 = (local % mt) * BT;
        ti.rows = min(BT, p.wg_rows - ti.row0);
        ti.row_end = p.wg_rows;
        ti.first = p.offsets[lo];
        ti.nkb = S.prefix[lo + 1] - S.prefix[lo];
    } else if (SWAP) {
        // an expert's tokens in mt tiles of equal size (a multiple of 16),
        // rather than full tiles and a small remainder that would still
        // stream the whole weight tile
        const int cnt = ti.row_end - p.offsets[lo];
        const int ts = ((cnt + mt - 1) / mt + 15) & ~15;
        ti.row0 = p.offsets[lo] + (local % mt) * ts;
        ti.rows = min(ts, ti.row_end - ti.row0);
    } else {
        ti.row0 = p.offsets[lo] + (local % mt) * BM;
        ti.rows = 0;
    }
    ti.col0 = (local / mt) * (SWAP ? (p.half ? kSwapFeatSwiglu : kSwapFeatStore) : (p.half ? BN / 2 : BN));
    if (SWAP && p.half && !WG) ti.half = p.half - ti.col0 <= kSwapFeatSwiglu / 2;
    else if (SWAP && !p.half && !p.fc && !WG) ti.half = p.N - ti.col0 <= kSwapFeatStore / 2;
    return ti;
}

__device__ __forceinline__ void fail(Shared& S, const Params& p) {
    S.abort_flag = 1;
    moe::raise_device_error(p.err, MOE_DEVERR_TIMEOUT);
}

__device__ __forceinline__ uint32_t bar(uint64_t& b) { return moe::smem_u32(&b); }

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// 32 consecutive fp32 values -> bf16, stored as four 16-byte vectors whose
// columns lie below ncols (ncols is a multiple of 8).
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* row, int col, int ncols, const float* v) {
    uint4* dst = reinterpret_cast<uint4*>(row + col);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if (col + 8 * i < ncols)
            dst[i] = make_uint4(moe::pack_bf16x2(v[8 * i], v[8 * i + 1]),
                                moe::pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                                moe::pack_bf16x2(v[8 * i + 4], v[8 * i + 5]),
                                moe::pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
}

__device__ __forceinline__ uint32_t quant4(float a, float b, float c, float d, float s) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(__fdiv_rn(a, s), __fdiv_rn(b, s)), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(__fdiv_rn(c, s), __fdiv_rn(d, s)), __NV_SATFINITE, __NV_E4M3);
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// FP8 promotion of one 64-column chunk of a k-block partial into the fp32
// accumulators a[]: store layout -> a[c*64 .. c*64+63] += s0 * (x0 | x1);
// SwiGLU layout -> gate a[c*32 ..] += s0 * x0 and up a[64 + c*32 ..] += s1 * x1.
__device__ __forceinline__ void ffma2(float& a0, float& a1, float s, uint32_t v0, uint32_t v1) {
    asm("{\n\t.reg .b64 acc, sv, vv;\n\t"
        "mov.b64 acc, {%0, %1};\n\t"
        "mov.b64 sv, {%2, %2};\n\t"
        "mov.b64 vv, {%3, %4};\n\t"
        "fma.rn.f32x2 acc, sv, vv, acc;\n\t"
        "mov.b64 {%0, %1}, acc;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(s), "r"(v0), "r"(v1));
}

template <int EPI>
__device__ __forceinline__ void promote_chunk(float (&a)[128], int c, float s0, float s1,
                                              const uint32_t (&x0)[32], const uint32_t (&x1)[32]) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        if (EPI == EPI_STORE) {
            ffma2(a[c * 64 + i], a[c * 64 + i + 1], s0, x0[i], x0[i + 1]);
            ffma2(a[c * 64 + 32 + i], a[c * 64 + 33 + i], s0, x1[i], x1[i + 1]);
        } else {
            ffma2(a[c * 32 + i], a[c * 32 + i + 1], s0, x0[i], x0[i + 1]);
            ffma2(a[64 + c * 32 + i], a[64 + c * 32 + i + 1], s1, x1[i], x1[i + 1]);
        }
    }
}

// ---------------------------------------------------------------- roles
// The producer and MMA roles run on a whole warp: every lane tracks the ring
// and polls the barriers, and one elected lane issues (see moe::elect_one).
template <bool FP8, int EPI>
__device__ void producer(const CUtensorMap* tmA, const CUtensorMap* tmB, uint8_t* stages,
                         Shared& S, const Params& p, int total) {
    int stage = 0;
    uint32_t phase = 0, issued = 0, issued_par = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
        const Tile ti = decode_tile<false>(t, S, p);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
            const bool got = moe::mbar_wait(bar(S.empty[stage]), phase ^ 1u, &S.abort_flag, kWaitNs);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            const uint32_t fb = bar(S.full[stage]);
            const uint32_t sa = moe::smem_u32(stages + stage * Geo<false, EPI>::kStageBytes);
            const uint32_t sb = sa + kStageA;
            const int kc = kb * (FP8 ? 128 : 64);
            if (moe::elect_one()) {
                moe::mbar_arrive_expect_tx(fb, Geo<false, EPI>::kStageBytes);
                moe::tma_load_2d(sa, tmA, fb, kc, ti.row0);
                if (EPI == EPI_STORE) {
                    moe::tma_load_3d(sb, tmB, fb, kc, ti.col0, ti.e);
                } else {
                    moe::tma_load_4d(sb, tmB, fb, kc, ti.col0, 0, ti.e);
                    moe::tma_load_4d(sb + (BN / 2) * 128, tmB, fb, kc, ti.col0, 1, ti.e);
                }
            }
            __syncwarp();
            issued |= 1u << stage;
            issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
            if (++stage == Geo<false, EPI>::kStages) { stage = 0; phase ^= 1u; }
        }
    }
    if (!ok && moe::elect_one()) {
        fail(S, p);
        int zero = 0;
        for (int s = 0; s < Geo<false, EPI>::kStages; ++s)
            if ((issued >> s) & 1u)
                moe::mbar_wait(bar(S.full[s]), (issued_par >> s) & 1u, &zero, kDrainNs);
    }
    __syncwarp();
}

// Token rows of a swapped tile (at most BT; the MMA's N is this rounded up to 16,
// which cta_group::2 M = 256 MMAs allow).
__device__ __forceinline__ int swap_rows(const Tile& ti) { return ti.rows; }
// MMA N of a swapped tile: the tokens rounded up to 16 (M = 256) or 32 (M = 128)
__device__ __forceinline__ int swap_n(const Tile& ti) { return ti.half ? (ti.rows + 31) & ~31 : (ti.rows + 15) & ~15; }

// Tile loop bounds: a CTA pair walks the tile list as one unit.
template <bool PAIR>
__device__ __forceinline__ int tile_first() { return PAIR ? blockIdx.x >> 1 : blockIdx.x; }
template <bool PAIR>
__device__ __forceinline__ int tile_step() { return PAIR ? gridDim.x >> 1 : gridDim.x; }

// Producer with swapped operands on a CTA pair (bf16).  Per k-block each CTA
// loads its 128 weight rows into the A region and its N/2 token rows into
// the B region, all counted on the leading CTA's full barrier (the leader
// posts both CTAs' bytes).  SwiGLU: CTA r's 128 weight rows are its 64
// features' gate and up rows, interleaved in groups of 8 (one 5-D box; an
// M = 128 tile takes 4 groups, 32 features, from tmW64).
// Tokens: one box of exactly the tile's N/2 rows (a multiple of 8, one
// tensor map per height).  A TMA instruction costs the issuing thread many
// cycles, so a k-block takes as few as possible.
template <int EPI, bool WG>
__device__ void producer_swap(const TokenMaps* tmX, const CUtensorMap* tmW, const CUtensorMap* tmW64,
                              uint8_t* stages, Shared& S, const Params& p, int total, uint32_t rank) {
    int stage = 0;
    uint32_t phase = 0, issued = 0, issued_par = 0;
    bool ok = true;
    for (int t = tile_first<true>(); ok && t < total; t += tile_step<true>()) {
        const Tile ti = decode_tile<true, WG>(t, S, p);
        const int nh = swap_n(ti) / 2;                 // token rows in each CTA: 8 .. 128
        const CUtensorMap* tmXh = &tmX->m[nh / 8 - 1];
        const int xrow = ti.row0 + static_cast<int>(rank) * nh;
        // weight gradient: this CTA's nh columns of dC in one or two 64-wide boxes
        const int xbytes = WG ? (nh > 64 ? 2 : 1) * 8192 : nh * 128;
        const int abytes = ti.half ? kStageA / 2 : kStageA;   // M = 128: 64 weight rows per CTA
        const int nkb = WG ? ti.nkb : p.k_blocks;
        const int nfull = WG ? (p.offsets[ti.e + 1] - ti.first) / 64 : 0;   // k-blocks read in place
        for (int kb = 0; kb < nkb; ++kb) {
            const bool got = moe::mbar_wait(bar(S.empty[stage]), phase ^ 1u, &S.abort_flag, kWaitNs);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            const uint32_t fb = moe::map_to_cta(bar(S.full[stage]), 0);
            const uint32_t sa = moe::smem_u32(stages + stage * Geo<true, EPI>::kStageBytes);
            const uint32_t sb = sa + kStageA;
            const int kc = kb * 64;
            if (moe::elect_one()) {
                if (rank == 0) moe::mbar_arrive_expect_tx(bar(S.full[stage]), 2 * (abytes + xbytes));
                if (WG) {
                    // weight gradient: A's 128 features and dC's nh columns of
                    // this CTA over 64 rows, as 64 x 64 MN-major swizzle atoms
                    // 8 KB apart, from the expert's own rows or, for its
                    // partial last k-block, from the zero-padded tails
                    const bool in_place = kb < nfull;
                    const CUtensorMap* ma = &tmX->m[in_place ? kWgA : kWgTailA];
                    const CUtensorMap* mc = &tmX->m[in_place ? kWgC : kWgTailC];
                    const int row = in_place ? ti.first + kc : ti.e * 64;
                    const int f0 = ti.col0 + static_cast<int>(rank) * 128;
                    moe::tma_load_2d_pair(sa, ma, fb, f0, row);
                    moe::tma_load_2d_pair(sa + 8192, ma, fb, f0 + 64, row);
                    moe::tma_load_2d_pair(sb, mc, fb, xrow, row);
                    if (nh > 64) moe::tma_load_2d_pair(sb + 8192, mc, fb, xrow + 64, row);
                } else if (EPI == EPI_STORE && p.mn_a) {
                    // two 64-feature x 64-row swizzle atoms, 8 KB apart (one for M = 128)
                    const int f0 = ti.col0 + static_cast<int>(rank) * (ti.half ? 64 : 128);
                    moe::tma_load_3d_pair(sa, tmW, fb, f0, kc, ti.e);
                    if (!ti.half) moe::tma_load_3d_pair(sa + 8192, tmW, fb, f0 + 64, kc, ti.e);
                } else if (EPI == EPI_STORE && ti.half) {   // 64 weight rows
                    moe::tma_load_3d_pair(sa, tmW64, fb, kc, ti.col0 + static_cast<int>(rank) * 64, ti.e);
                } else if (EPI == EPI_STORE) {
                    moe::tma_load_3d_pair(sa, tmW, fb, kc, ti.col0 + static_cast<int>(rank) * 128, ti.e);
                } else if (ti.half) {   // 4 groups: this CTA's 32 features
                    moe::tma_load_5d_pair(sa, tmW64, fb, kc, 0, 0, (ti.col0 + static_cast<int>(rank) * 32) / 8, ti.e);
                } else {   // 8 groups of (8 gate rows, 8 up rows) of this CTA's 64 features
                    moe::tma_load_5d_pair(sa, tmW, fb, kc, 0, 0, (ti.col0 + static_cast<int>(rank) * 64) / 8, ti.e);
                }
                if (!WG) moe::tma_load_2d_pair(sb, tmXh, fb, kc, xrow);
            }
            __syncwarp();
            issued |= 1u << stage;
            issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
            if (++stage == Geo<true, EPI>::kStages) { stage = 0; phase ^= 1u; }
        }
    }
    if (!ok && moe::elect_one()) {
        fail(S, p);
        int zero = 0;
        if (rank == 0) {
            for (int s = 0; s < Geo<true, EPI>::kStages; ++s)
                if ((issued >> s) & 1u)
                    moe::mbar_wait(bar(S.full[s]), (issued_par >> s) & 1u, &zero, kDrainNs);
        } else {
            // the peer's loads complete on the leader's barrier: give them time to land
            const uint64_t t0 = moe::global_timer_ns();
            while (moe::global_timer_ns() - t0 < 1000000ull) __nanosleep(1000);
        }
    }
    __syncwarp();
}

// Source token of row `row` of the permuted order, or -1 when the row is past
// the tile's expert or its slot is out of range (that case is reported).
__device__ __forceinline__ int gather_token(const Params& p, int row, int row_end, bool report) {
    if (row >= row_end) return -1;
    const int slot = p.sorted_rows[row];
    const int t = slot >= 0 ? slot / p.topk : -1;
    if (t < 0 || t >= p.T) {
        if (report) moe::raise_device_error(p.err, MOE_DEVERR_ROUTE);
        return -1;
    }
    return t;
}

// Producer for gathered A, run by issuing warp g (0 = warp 0, which also
// posts the stage's byte count and loads the weight tile).  The warp reads the
// tile's 128 tokens; then its lane 0 waits for each stage and gathers rows
// 4j..4j+3 for j = g, g + kGatherWarps, ... below the tile's live rows.
// Gathered bytes may land before warp 0 posts the count: the barrier's
// transaction count goes negative until then, and the phase cannot complete
// before warp 0's arrival.  A row without a token inside a fetched quad (past
// the expert's end, or an out-of-range slot) is fetched from token 0, so every
// coordinate stays inside the tensor; the epilogue never stores such a row.
template <bool FP8, int EPI>
__device__ void producer_gather(const CUtensorMap* tmA, const CUtensorMap* tmB, uint8_t* stages,
                                Shared& S, const Params& p, int total, int g) {
    const int lane = threadIdx.x & 31;
    int* gtok = aux(S).gtok[g];
    int stage = 0;
    uint32_t phase = 0, issued = 0, issued_par = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
        const Tile ti = decode_tile<false>(t, S, p);
        __syncwarp();  // lane 0 is done with the previous tile's tokens
#pragma unroll
        for (int j = 0; j < BM / 32; ++j) {
            const int tok = gather_token(p, ti.row0 + lane + 32 * j, ti.row_end, g == 0);
            gtok[lane + 32 * j] = tok >= 0 ? tok : 0;
        }
        __syncwarp();
        // only the quads that hold a live row are fetched; the rest of the A
        // tile keeps stale bytes, which only feed rows the epilogue drops
        const int nq = (min(BM, ti.row_end - ti.row0) + 3) / 4;
        if (lane == 0) {
            for (int kb = 0; kb < p.k_blocks; ++kb) {
                if (!moe::mbar_wait(bar(S.empty[stage]), phase ^ 1u, &S.abort_flag, kWaitNs)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = bar(S.full[stage]);
                const uint32_t sa = moe::smem_u32(stages + stage * Geo<false, EPI>::kStageBytes);
                const int kc = kb * (FP8 ? 128 : 64);
                if (g == 0) {
                    moe::mbar_arrive_expect_tx(fb, kStageB + nq * 512);
                    const uint32_t sb = sa + kStageA;
                    if (EPI == EPI_STORE) {
                        moe::tma_load_3d(sb, tmB, fb, kc, ti.col0, ti.e);
                    } else {
                        moe::tma_load_4d(sb, tmB, fb, kc, ti.col0, 0, ti.e);
                        moe::tma_load_4d(sb + (BN / 2) * 128, tmB, fb, kc, ti.col0, 1, ti.e);
                    }
                }
                // token quads are read four at a time before their gathers
                // are issued, so the shared-memory loads overlap instead of
                // each waiting behind the previous gather (16 registers)
                constexpr int NQ = (BM / 4 + kGatherWarps - 1) / kGatherWarps, CH = 4;
#pragma unroll
                for (int c = 0; c < NQ; c += CH) {
                    int4 r[CH];
#pragma unroll
                    for (int i = 0; i < CH; ++i) {
                        const int j = g + (c + i) * kGatherWarps;
                        r[i] = c + i < NQ && j < nq ? *reinterpret_cast<const int4*>(gtok + 4 * j)
                                                    : make_int4(0, 0, 0, 0);
                    }
#pragma unroll
                    for (int i = 0; i < CH; ++i) {
                        const int j = g + (c + i) * kGatherWarps;
                        if (c + i < NQ && j < nq)
                            moe::tma_gather4(sa + j * 512, tmA, fb, kc, r[i].x, r[i].y, r[i].z, r[i].w);
                    }
                }
                issued |= 1u << stage;
                issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
                if (++stage == Geo<false, EPI>::kStages) { stage = 0; phase ^= 1u; }
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (!ok && lane == 0) {
        fail(S, p);
        // this warp's gathers land whatever the other roles do; the phases
        // they count towards may never complete, so each wait is short
        int zero = 0;
        for (int s = 0; s < Geo<false, EPI>::kStages; ++s)
            if ((issued >> s) & 1u)
                moe::mbar_wait(bar(S.full[s]), (issued_par >> s) & 1u, &zero, kDrainNs);
    }
}

template <bool FP8, int EPI, bool SWAP, bool WG>
__device__ void mma_issuer(uint8_t* stages, Shared& S, const Params& p, int total, uint32_t tmem) {
    uint32_t idesc = moe::make_idesc(FP8 ? 0u : 1u, BM, BN);
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true, issued = false;
    for (int t = tile_first<SWAP>(); ok && t < total; t += tile_step<SWAP>()) {
        if (SWAP) {
            const Tile ti = decode_tile<true, WG>(t, S, p);
            const int n = swap_n(ti);
            const int m = ti.half ? BM : 2 * BM;
            idesc = WG ? moe::make_idesc_ab_mn(1u, 2 * BM, n)
                 : EPI == EPI_STORE && p.mn_a ? moe::make_idesc_a_mn(1u, m, n) : moe::make_idesc(1u, m, n);
        }
        if (!FP8) {
            // with a pair, the peer's epilogue arrives here from the other CTA
            const bool got = SWAP ? moe::mbar_wait_cluster(bar(S.acc_empty[acc]), acc_phase ^ 1u, &S.abort_flag, kWaitNs)
                                  : moe::mbar_wait(bar(S.acc_empty[acc]), acc_phase ^ 1u, &S.abort_flag, kWaitNs);
            if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
            moe::tc_fence_after();
        }
        // weight-gradient tiles of an expert without rows have no k-blocks:
        // the accumulator is committed untouched and the epilogue writes zeros
        const int nkb = WG ? decode_tile<SWAP, WG>(t, S, p).nkb : p.k_blocks;
        for (int kb = 0; kb < nkb; ++kb) {
            if (FP8) {
                const bool got = moe::mbar_wait(bar(S.acc_empty[acc]), acc_phase ^ 1u, &S.abort_flag, kWaitNs);
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                moe::tc_fence_after();
            }
            const bool got = moe::mbar_wait(bar(S.full[stage]), phase, &S.abort_flag, kWaitNs);
            if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
            moe::tc_fence_after();
            const uint32_t sa = moe::smem_u32(stages + stage * Geo<SWAP, EPI>::kStageBytes);
            // MN-major operands (the data gradient's weights; both operands of
            // the weight gradient): a K step of 16 rows is 2 KB further on;
            // K-major: 32 bytes
            const bool amn = WG || (SWAP && EPI == EPI_STORE && p.mn_a);
            const uint64_t adesc = amn ? moe::smem_desc_sw128_mn(sa, 8192) : moe::smem_desc_sw128(sa);
            const uint64_t astep = amn ? 2048 >> 4 : 2;
            const uint64_t bdesc = WG ? moe::smem_desc_sw128_mn(sa + kStageA, 8192) : moe::smem_desc_sw128(sa + kStageA);
            const uint64_t bstep = WG ? 2048 >> 4 : 2;
            const uint32_t d = tmem + static_cast<uint32_t>(acc * BN);
            // the same (lowest) lane is elected every time, so its commits
            // track all the MMAs it issued
            if (moe::elect_one()) {
#pragma unroll
                for (int k = 0; k < 4; ++k)  // 32 bytes of K per instruction; +2 = +32 B start address
                    if (FP8)
                        moe::mma_fp8(d, adesc + 2 * k, bdesc + 2 * k, idesc, k > 0);
                    else if (SWAP)
                        moe::mma_bf16_pair(d, adesc + astep * k, bdesc + bstep * k, idesc, (kb | k) != 0);
                    else
                        moe::mma_bf16(d, adesc + 2 * k, bdesc + 2 * k, idesc, (kb | k) != 0);
                if (SWAP) moe::tc_commit_pair(bar(S.empty[stage]), 0x3);   // frees the stage in both CTAs
                else moe::tc_commit(bar(S.empty[stage]));
                if (FP8) moe::tc_commit(bar(S.acc_full[acc]));
            }
            __syncwarp();
            issued = true;
            if (++stage == Geo<SWAP, EPI>::kStages) { stage = 0; phase ^= 1u; }
            if (FP8) {
                acc ^= 1;
                if (!acc) acc_phase ^= 1u;
            }
        }
        if (!ok) break;
        if (!FP8) {
            if (moe::elect_one()) {
                if (SWAP) moe::tc_commit_pair(bar(S.acc_full[acc]), 0x3);
                else moe::tc_commit(bar(S.acc_full[acc]));
            }
            __syncwarp();
            acc ^= 1;
            if (!acc) acc_phase ^= 1u;
        }
    }
    if (!ok && moe::elect_one()) fail(S, p);
    __syncwarp();
    if (issued) {  // every MMA of this CTA (pair) has finished before TMEM is freed
        int zero = 0;
        if (moe::elect_one()) {
            if (SWAP) moe::tc_commit_pair(bar(S.mma_done), 0x1);
            else moe::tc_commit(bar(S.mma_done));
        }
        __syncwarp();
        moe::mbar_wait(bar(S.mma_done), 0, &zero, kDrainNs);
    }
}

// Fused weighted combine, one 16-byte chunk (8 features) of token t's
// 128-feature block at f0: out[t, f] = sum over live slots j, in slot order,
// of w[t, j] * Y2[row_pos[t*k + j], f], accumulated in fp32 with fmaf exactly
// as moe_combine does, rounded to bf16.  The rows come through L2 (other
// CTAs stored most of them).
__device__ __forceinline__ void combine_chunk(const Params& p, int t, int f0, int c) {
    const int f = f0 + 8 * c;
    if (f >= p.out_cols) return;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    const __nv_bfloat16* Y2 = static_cast<const __nv_bfloat16*>(p.out);
    // up to eight slots at a time: their rows are all requested before the
    // first is summed, so the loads are in flight together
    constexpr int G = 8;
    for (int j0 = 0; j0 < p.topk; j0 += G) {
        uint4 v[G];
        float wj[G];
        bool use[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int j = j0 + g;
            use[g] = false;
            wj[g] = 0.0f;
            v[g] = make_uint4(0, 0, 0, 0);
            if (j < p.topk) {
                const int64_t slot = static_cast<int64_t>(t) * p.topk + j;
                if (p.ids[slot] != p.E) {
                    const int pos = p.row_pos[slot];
                    if (pos < 0 || pos >= p.M_cap) {
                        moe::raise_device_error(p.err, MOE_DEVERR_ROUTE);
                    } else {
                        use[g] = true;
                        wj[g] = p.wts[slot];
                        v[g] = __ldcg(reinterpret_cast<const uint4*>(Y2 + static_cast<int64_t>(pos) * p.out_cols + f));
                    }
                }
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            if (!use[g]) continue;
            const uint32_t v4[4] = {v[g].x, v[g].y, v[g].z, v[g].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] = fmaf(wj[g], moe::bf16_lo(v4[i]), acc[2 * i]);
                acc[2 * i + 1] = fmaf(wj[g], moe::bf16_hi(v4[i]), acc[2 * i + 1]);
            }
        }
    }
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.cout) + static_cast<int64_t>(t) * p.out_cols + f;
    *reinterpret_cast<uint4*>(out) = make_uint4(moe::pack_bf16x2(acc[0], acc[1]), moe::pack_bf16x2(acc[2], acc[3]),
                                                moe::pack_bf16x2(acc[4], acc[5]), moe::pack_bf16x2(acc[6], acc[7]));
}

// After a swapped store tile: every epilogue thread of the CTA has stored
// its rows of the tile (and fenced them; a bounded mbarrier wait, not a
// hardware barrier, so that a CTA winding down after a timeout cannot hang
// it); then each token of the tile bumps
// the counter of its (token, 128-feature block).  The thread that brings it
// to the token's number of live slots holds the last of them: its warp sums
// that token's block (two tokens at a time, 16 lanes each) and resets the
// counter.  Every (token, block) is summed once, in slot order, whichever CTA
// stores last, so the result is the same bits as moe_combine's.
__device__ __forceinline__ bool fused_combine_tile(Shared& S, const Params& p, const Tile& ti, uint32_t rank,
                                                   uint32_t& cph) {
    __threadfence();
    moe::mbar_arrive(bar(S.cbar));
    if (!moe::mbar_wait(bar(S.cbar), cph, &S.abort_flag, kWaitNs)) return false;
    cph ^= 1u;
    const int f0 = ti.col0 + static_cast<int>(rank) * 128;
    if (f0 >= p.out_cols) return true;
    const int fb = f0 / 128;
    const int et = threadIdx.x - 128, lane = threadIdx.x & 31;
    int t = 0;
    bool last = false;
    if (et < ti.rows) {
        const int slot = p.sorted_rows[ti.row0 + et];
        t = slot / p.topk;
        if (t >= 0 && t < p.T) {
            int live = 0;
            for (int j = 0; j < p.topk; ++j) live += p.ids[static_cast<int64_t>(t) * p.topk + j] != p.E;
            int* c = p.counters + static_cast<int64_t>(t) * p.nfb + fb;
            last = atomicAdd(c, 1) == live - 1;
            if (last) *c = 0;   // no other slot of this token touches it in this call
        } else {
            moe::raise_device_error(p.err, MOE_DEVERR_ROUTE);
        }
    }
    unsigned mask = __ballot_sync(0xffffffffu, last);
    if (mask) __threadfence();   // the other contributors' rows are visible from here on
    while (mask) {
        const int a = __ffs(mask) - 1;
        mask &= mask - 1;
        int b = -1;
        if (mask) {
            b = __ffs(mask) - 1;
            mask &= mask - 1;
        }
        const int ta = __shfl_sync(0xffffffffu, t, a);
        const int tb = __shfl_sync(0xffffffffu, t, b < 0 ? a : b);
        if (lane < 16) combine_chunk(p, ta, f0, lane);
        else if (b >= 0) combine_chunk(p, tb, f0, lane - 16);
    }
    return true;
}

// Tokens whose slots are all sentinels get no contribution: their output
// rows are zeros (spread over every epilogue thread of the grid).
__device__ void fused_combine_empty_tokens(const Params& p) {
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kEpiThreads + (threadIdx.x - 128);
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * kEpiThreads;
    for (int64_t t = tid; t < p.T; t += nthr) {
        bool any = false;
        for (int j = 0; j < p.topk; ++j) any |= p.ids[t * p.topk + j] != p.E;
        if (any) continue;
        uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.cout) + t * p.out_cols);
        for (int v = 0; v < p.out_cols / 8; ++v) o[v] = make_uint4(0, 0, 0, 0);
    }
}

// Store M = 128 tile (forward and data gradient): lane l of this CTA holds
// weight row (output feature) l % 64 for token (l / 64) * nh + column, columns
// below nh = N/2.  Each half of the epilogue takes 64 columns.
__device__ __forceinline__ void store_half_tile(const Params& p, const Tile& ti, uint32_t ta, int q, int hsel,
                                                int lane, uint32_t rank) {
    const int nh = swap_n(ti) / 2, tok0 = (q >> 1) * nh, ntok = ti.rows;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    const int f = ti.col0 + static_cast<int>(rank) * 64 + (q & 1) * 32 + lane;
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
        const int col = hsel * 64 + c * 32;
        if (col >= nh || tok0 + col >= ntok) break;   // the same for the whole warp
        const int jmax = min(32, min(nh - col, ntok - tok0 - col));   // token columns of the chunk
        uint32_t v[32];
        moe::tmem_ld32(ta + col, v);
        moe::tmem_ld_wait();
        if (f < p.out_cols) {
            __nv_bfloat16* o = out + static_cast<int64_t>(ti.row0 + tok0 + col) * p.out_cols + f;
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < jmax) o[static_cast<int64_t>(j) * p.out_cols] = __float2bfloat16_rn(__uint_as_float(v[j]));
        }
    }
}

// SwiGLU M = 128 tile: lane l of this CTA holds weight row l % 64 (its 32
// features' gate and up rows, interleaved in groups of 8 as in a full tile)
// for token (l / 64) * nh + column, columns below nh = N/2.  Each half of the
// epilogue takes 64 columns; gate and up lanes swap halves of each 32-column
// chunk as in a full tile.
__device__ __forceinline__ void swiglu_half_tile(const Params& p, const Tile& ti, uint32_t ta, int q, int hsel,
                                                 int lane, uint32_t rank) {
    const int nh = swap_n(ti) / 2, tok0 = (q >> 1) * nh, ntok = ti.rows;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
        const int col = hsel * 64 + c * 32;
        if (col >= nh || tok0 + col >= ntok) break;   // the same for the whole warp
        const int jmax = min(32, min(nh - col, ntok - tok0 - col));   // token columns of the chunk
        uint32_t v[32];
        moe::tmem_ld32(ta + col, v);
        moe::tmem_ld_wait();
        const int r = (lane >> 3) & 1;   // 0: gate lane, 1: up lane
        float h[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float lo = __uint_as_float(v[j]), hi = __uint_as_float(v[16 + j]);
            const float o = __shfl_xor_sync(0xffffffffu, r ? lo : hi, 8);
            h[j] = r ? silu_mul(o, hi) : silu_mul(lo, o);
        }
        const int f = ti.col0 + static_cast<int>(rank) * 32 + 16 * (q & 1) + 8 * (lane >> 4) + (lane & 7);
        const int t0 = 16 * r;   // within the chunk
        if (f < p.out_cols) {
            __nv_bfloat16* o = out + static_cast<int64_t>(ti.row0 + tok0 + col + t0) * p.out_cols + f;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (t0 + j < jmax) o[static_cast<int64_t>(j) * p.out_cols] = __float2bfloat16_rn(h[j]);
        }
    }
}

template <bool FP8, int EPI, bool SWAP, bool WG>
__device__ void epilogue(Shared& S, const Params& p, int total, uint32_t tmem, uint32_t rank) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;               // TMEM lane quarter this warp may access
    const int hsel = (warp - 4) >> 2;     // which half of the tile's columns
    const int r = q * 32 + lane;          // accumulator row of this thread
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    int acc = 0, xsel = 0;
    uint32_t acc_phase = 0, xphase = 0;
    uint32_t cph = 0;                    // fused combine barrier phase
    const int KB = p.k_blocks;

    // the pair's MMA waits for both CTAs' epilogues on the leader's barrier
    uint32_t acc_empty_leader[2] = {0, 0};
    if (SWAP) {
        acc_empty_leader[0] = moe::map_to_cta(bar(S.acc_empty[0]), 0);
        acc_empty_leader[1] = moe::map_to_cta(bar(S.acc_empty[1]), 0);
    }
    for (int t = tile_first<SWAP>(); t < total; t += tile_step<SWAP>()) {
        const Tile ti = decode_tile<SWAP, WG>(t, S, p);
        const int row = ti.row0 + r;
        const bool live = row < ti.row_end;
        if (SWAP) {
            // accumulator lane = weight row, column = token of the tile
            if (!moe::mbar_wait(bar(S.acc_full[acc]), acc_phase, &S.abort_flag, kWaitNs)) { fail(S, p); return; }
            moe::tc_fence_after();
            const uint32_t ta = lane_base + static_cast<uint32_t>(acc * BN);
            const int ntok = swap_rows(ti);
            // weight gradient: expert e's output rows start at e * wg_rows
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) +
                                 (WG ? static_cast<int64_t>(ti.e) * p.wg_rows * p.out_cols : 0);
            if (EPI != EPI_STORE && ti.half) {
                swiglu_half_tile(p, ti, ta, q, hsel, lane, rank);
            } else if (EPI == EPI_STORE && ti.half) {
                store_half_tile(p, ti, ta, q, hsel, lane, rank);
            } else {
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    const int col = hsel * 128 + c * 32;
                    if (col >= ntok) break;                       // the same for the whole warp
                    uint32_t v[32];
                    if (!WG || ti.nkb > 0) {
                        moe::tmem_ld32(ta + col, v);
                        moe::tmem_ld_wait();
                    } else {   // an expert without rows: its weight gradient is zero
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0u;
                    }
                    if (EPI == EPI_STORE) {
                        // one output feature per lane; a warp store covers 64
                        // contiguous bytes of one token row
                        const int f = ti.col0 + static_cast<int>(rank) * 128 + q * 32 + lane;
                        if (f < p.out_cols) {
                            __nv_bfloat16* o = out + static_cast<int64_t>(ti.row0 + col) * p.out_cols + f;
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (col + j < ntok) o[static_cast<int64_t>(j) * p.out_cols] = __float2bfloat16_rn(__uint_as_float(v[j]));
                        }
                    } else {
                        // lane l holds the gate (up, if bit 3 of l is set) row of
                        // feature 16q + 8(l / 16) + l % 8; lanes l and l ^ 8 share
                        // a feature.  The gate lane computes the chunk's first 16
                        // tokens, the up lane the last 16, each receiving the
                        // other's values for its tokens.
                        const int r = (lane >> 3) & 1;            // 0: gate lane, 1: up lane
                        float h[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float lo = __uint_as_float(v[j]), hi = __uint_as_float(v[16 + j]);
                            const float o = __shfl_xor_sync(0xffffffffu, r ? lo : hi, 8);
                            h[j] = r ? silu_mul(o, hi) : silu_mul(lo, o);
                        }
                        const int f = ti.col0 + static_cast<int>(rank) * 64 + 16 * q + 8 * (lane >> 4) + (lane & 7);
                        const int t0 = col + 16 * r;
                        if (f < p.out_cols) {
                            __nv_bfloat16* o = out + static_cast<int64_t>(ti.row0 + t0) * p.out_cols + f;
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (t0 + j < ntok) o[static_cast<int64_t>(j) * p.out_cols] = __float2bfloat16_rn(h[j]);
                        }
                    }
                }
            }
            moe::tc_fence_before();
            if (rank != 0) moe::mbar_arrive_cluster(acc_empty_leader[acc]);
            else moe::mbar_arrive(bar(S.acc_empty[acc]));
            acc ^= 1;
            if (!acc) acc_phase ^= 1u;
            if (EPI == EPI_STORE && p.fc && !fused_combine_tile(S, p, ti, rank, cph)) { fail(S, p); return; }
        } else if (!FP8) {
            if (!moe::mbar_wait(bar(S.acc_full[acc]), acc_phase, &S.abort_flag, kWaitNs)) { fail(S, p); return; }
            moe::tc_fence_after();
            const uint32_t ta = lane_base + static_cast<uint32_t>(acc * BN);
            __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(row) * p.out_cols;
            if (EPI == EPI_STORE) {
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t v[32];
                    moe::tmem_ld32(ta + hsel * 128 + c * 32, v);
                    moe::tmem_ld_wait();
                    if (live) store_bf16x32(orow, ti.col0 + hsel * 128 + c * 32, p.out_cols,
                                            reinterpret_cast<const float*>(v));
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    uint32_t g[32], u[32];
                    moe::tmem_ld32(ta + hsel * 64 + c * 32, g);
                    moe::tmem_ld32(ta + 128 + hsel * 64 + c * 32, u);
                    moe::tmem_ld_wait();
                    float h[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) h[i] = silu_mul(__uint_as_float(g[i]), __uint_as_float(u[i]));
                    if (live) store_bf16x32(orow, ti.col0 + hsel * 64 + c * 32, p.out_cols, h);
                }
            }
            moe::tc_fence_before();
            moe::mbar_arrive(bar(S.acc_empty[acc]));
            acc ^= 1;
            if (!acc) acc_phase ^= 1u;
        } else {
            float a[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) a[i] = 0.0f;
            const float* sb_row = p.b_scales + static_cast<int64_t>(ti.e) * p.nb_scale * KB;
            const int nb0 = EPI == EPI_STORE ? (ti.col0 + hsel * 128) / 128 : ti.col0 / 128;
            const int nb1 = EPI == EPI_STORE ? nb0 : (p.half + ti.col0) / 128;
            const bool nb_ok = nb0 < p.nb_scale;
            // activation scales of this row: group-major over permuted rows,
            // or row-major over tokens when A is gathered
            const float* sa_row;
            int sa_step;
            bool row_ok;
            if (p.gx) {
                const int tok = gather_token(p, row, ti.row_end, false);
                row_ok = tok >= 0;
                sa_row = p.a_scales + static_cast<int64_t>(row_ok ? tok : 0) * KB;
                sa_step = 1;
            } else {
                row_ok = row < p.M_cap;
                sa_row = p.a_scales + row;
                sa_step = p.M_cap;
            }
            // Block scales travel through a per-thread ring of kScaleRing slots
            // in shared memory, filled by 4-byte cp.async copies (one commit
            // group per k-block) about kScaleRing k-blocks before they are
            // used, so their global-load latency stays off the promotion's
            // critical path and they take no registers.  Layout [slot][value][thread] keeps
            // the accesses free of bank conflicts.
            constexpr int R = kScaleRing;
            const int et = threadIdx.x - 128;                 // epilogue thread 0..255
            float* ring = aux(S).scale_ring;
            auto prefetch = [&](int kq, int slot) {
                if (kq < KB) {
                    if (row_ok)
                        moe::cp_async4(moe::smem_u32(ring + (slot * 3 + 0) * kEpiThreads + et),
                                       sa_row + static_cast<int64_t>(kq) * sa_step);
                    if (nb_ok)
                        moe::cp_async4(moe::smem_u32(ring + (slot * 3 + 1) * kEpiThreads + et),
                                       sb_row + nb0 * KB + kq);
                    if (EPI != EPI_STORE)
                        moe::cp_async4(moe::smem_u32(ring + (slot * 3 + 2) * kEpiThreads + et),
                                       sb_row + nb1 * KB + kq);
                }
                moe::cp_async_commit();
            };
#pragma unroll
            for (int i = 0; i < R; ++i) prefetch(i, i);
            for (int kb = 0; kb < KB; ++kb) {
                const int slot = kb % R;
                moe::cp_async_wait<R - 1>();               // k-block kb's group has landed
                const float sa = row_ok ? ring[(slot * 3 + 0) * kEpiThreads + et] : 0.0f;
                const float sb0 = nb_ok ? ring[(slot * 3 + 1) * kEpiThreads + et] : 0.0f;
                const float sb1 = EPI != EPI_STORE ? ring[(slot * 3 + 2) * kEpiThreads + et] : 0.0f;
                const float s0 = sa * sb0;
                const float s1 = EPI == EPI_STORE ? s0 : sa * sb1;
                if (!moe::mbar_wait(bar(S.acc_full[acc]), acc_phase, &S.abort_flag, kWaitNs)) { fail(S, p); return; }
                moe::tc_fence_after();
                const uint32_t ta = lane_base + static_cast<uint32_t>(acc * BN);
                // Two chunks of 64 columns.  The TMEM buffer goes back to the
                // MMA as soon as the second chunk is in registers, before its
                // FMAs, to keep the promotion short on the MMA's critical path.
                // Paired FMAs (fma.rn.f32x2) round each lane exactly as fmaf.
                uint32_t x0[32], x1[32];
                if (EPI == EPI_STORE) {
                    moe::tmem_ld32(ta + hsel * 128, x0);
                    moe::tmem_ld32(ta + hsel * 128 + 32, x1);
                } else {
                    moe::tmem_ld32(ta + hsel * 64, x0);
                    moe::tmem_ld32(ta + 128 + hsel * 64, x1);
                }
                moe::tmem_ld_wait();
                promote_chunk<EPI>(a, 0, s0, s1, x0, x1);
                if (EPI == EPI_STORE) {
                    moe::tmem_ld32(ta + hsel * 128 + 64, x0);
                    moe::tmem_ld32(ta + hsel * 128 + 96, x1);
                } else {
                    moe::tmem_ld32(ta + hsel * 64 + 32, x0);
                    moe::tmem_ld32(ta + 128 + hsel * 64 + 32, x1);
                }
                moe::tmem_ld_wait();
                moe::tc_fence_before();
                moe::mbar_arrive(bar(S.acc_empty[acc]));
                acc ^= 1;
                if (!acc) acc_phase ^= 1u;
                // the next copies into this slot are issued once the buffer is
                // released: their issue cost stays off the MMA's critical path
                prefetch(kb + R, slot);
                promote_chunk<EPI>(a, 1, s0, s1, x0, x1);
            }
            moe::cp_async_wait<0>();
            if (EPI == EPI_STORE) {
                __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(row) * p.out_cols;
                if (live) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) store_bf16x32(orow, ti.col0 + hsel * 128 + c * 32, p.out_cols, a + c * 32);
                }
            } else if (EPI == EPI_SWIGLU) {
                __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(row) * p.out_cols;
#pragma unroll
                for (int i = 0; i < 64; ++i) a[i] = silu_mul(a[i], a[64 + i]);
                if (live) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) store_bf16x32(orow, ti.col0 + hsel * 64 + c * 32, p.out_cols, a + c * 32);
                }
            } else {
                // h rounded to bf16, then quantised per 128 columns; the two
                // threads holding a row's halves exchange their amax.
                float amax = 0.0f;
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    a[i] = __bfloat162float(__float2bfloat16_rn(silu_mul(a[i], a[64 + i])));
                    amax = fmaxf(amax, fabsf(a[i]));
                }
                aux(S).amax_x[xsel][hsel][r] = amax;
                moe::mbar_arrive(bar(S.xbar[xsel]));
                if (!moe::mbar_wait(bar(S.xbar[xsel]), xphase, &S.abort_flag, kWaitNs)) { fail(S, p); return; }
                amax = fmaxf(amax, aux(S).amax_x[xsel][hsel ^ 1][r]);
                xsel ^= 1;
                if (!xsel) xphase ^= 1u;
                const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
                if (live) {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) +
                                                          static_cast<int64_t>(row) * p.out_cols +
                                                          ti.col0 + hsel * 64);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const float* h = a + 16 * v;
                        dst[v] = make_uint4(quant4(h[0], h[1], h[2], h[3], s), quant4(h[4], h[5], h[6], h[7], s),
                                            quant4(h[8], h[9], h[10], h[11], s),
                                            quant4(h[12], h[13], h[14], h[15], s));
                    }
                    if (hsel == 0) p.out_scales[static_cast<int64_t>(ti.col0 / 128) * p.M_cap + row] = s;
                }
            }
        }
    }
}

// Sentinel rows [offsets[E], M_cap) of the output: zeros (q = 0 and scale 1
// for the quantising epilogue), spread over every epilogue thread of the grid.
template <int EPI>
__device__ void zero_sentinel_rows(const Params& p) {
    const int L = p.offsets[p.E];
    const int64_t rows = static_cast<int64_t>(p.M_cap) - L;
    if (rows <= 0) return;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kEpiThreads + (threadIdx.x - 128);
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * kEpiThreads;
    const int esz = EPI == EPI_SWIGLU_Q ? 1 : 2;
    const int64_t vpr = static_cast<int64_t>(p.out_cols) * esz / 16;
    uint4* base = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) + static_cast<int64_t>(L) * p.out_cols * esz);
    for (int64_t i = tid; i < rows * vpr; i += nthr) base[i] = make_uint4(0, 0, 0, 0);
    if (EPI == EPI_SWIGLU_Q) {
        const int G = p.out_cols / 128;
        for (int64_t i = tid; i < rows * G; i += nthr) {
            const int64_t g = i / rows, rr = i - g * rows;
            p.out_scales[g * p.M_cap + L + rr] = 1.0f;
        }
    }
}

template <bool FP8, int EPI, bool SWAP, bool WG = false>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ TokenMaps tmX,
                    const Params p) {
    static_assert(!(SWAP && FP8), "swapped operands are a bf16 path");
    const uint32_t rank = SWAP ? moe::cluster_ctarank() : 0;   // 0 leads a pair
    extern __shared__ uint8_t smem_raw[];
    uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Shared& S = *reinterpret_cast<Shared*>(stages + Geo<SWAP, EPI>::kStages * Geo<SWAP, EPI>::kStageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Geo<SWAP, EPI>::kStages; ++s) {
            moe::mbar_init(bar(S.full[s]), 1);
            moe::mbar_init(bar(S.empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            moe::mbar_init(bar(S.acc_full[a]), 1);
            moe::mbar_init(bar(S.acc_empty[a]), SWAP ? 2 * kEpiThreads : kEpiThreads);
            moe::mbar_init(bar(S.xbar[a]), kEpiThreads);
        }
        moe::mbar_init(bar(S.mma_done), 1);
        moe::mbar_init(bar(S.cbar), kEpiThreads);
        S.abort_flag = 0;
        moe::fence_barrier_init();
    }
    if (warp == 0) {
        // validate offsets and build the row-tile prefix (8 experts per lane)
        int mt[8], kbl[8], sum = 0, ksum = 0, bad = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane * 8 + i;
            mt[i] = 0;
            kbl[i] = 0;
            if (e < p.E) {
                const int lo = p.offsets[e], hi = p.offsets[e + 1];
                if (hi < lo) bad = 1;
                constexpr int RT = SWAP ? BT : BM;   // rows of an expert per tile
                mt[i] = hi > lo ? (hi - lo + RT - 1) / RT : 0;
                if (WG) kbl[i] = hi > lo ? (hi - lo + 63) / 64 : 0;   // k-blocks of its rows
                ksum += kbl[i];
                sum += mt[i];
            }
        }
        if (lane == 0 && (p.offsets[0] != 0 || p.offsets[p.E] > p.M_cap)) bad = 1;
        // gathered A: sorted_rows holds T * topk entries
        if (lane == 0 && p.gx && p.offsets[p.E] > p.T * p.topk) bad = 1;
        bad = __any_sync(0xffffffffu, bad);
        int incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        int run = incl - sum;
        if (!WG) {   // the weight gradient keeps its k-block prefix here instead
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = lane * 8 + i;
                if (e < p.E) { S.prefix[e] = run; run += mt[i]; }
            }
            if (lane == 31) S.prefix[p.E] = incl;
        }
        if (WG) {
            int kincl = ksum;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, kincl, off);
                if (lane >= off) kincl += o;
            }
            int krun = kincl - ksum;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = lane * 8 + i;
                if (e < p.E) { S.prefix[e] = krun; krun += kbl[i]; }
            }
            if (lane == 31) S.prefix[p.E] = kincl;
        }
        if (lane == 0) {
            S.valid = !bad;
            if (bad && blockIdx.x == 0) moe::raise_device_error(p.err, MOE_DEVERR_OFFSETS);
        }
    } else if (warp == 1 && lane == 0) {
        moe::prefetch_tensormap(&tmA);
        moe::prefetch_tensormap(&tmB);
        if (SWAP) {
            for (int j = 0; j < (WG ? kWgMaps : kTokenMaps); ++j) moe::prefetch_tensormap(&tmX.m[j]);
        }
    }
    __syncthreads();
    if (!S.valid) return;   // both CTAs of a pair read the same offsets and leave together
    if (warp == 1) {
        if (SWAP) {
            moe::tmem_alloc_pair(moe::smem_u32(&S.tmem_base), kTmemCols);
            moe::tmem_relinquish_pair();
        } else {
            moe::tmem_alloc(moe::smem_u32(&S.tmem_base), kTmemCols);
            moe::tmem_relinquish();
        }
    }
    moe::tc_fence_before();
    if (SWAP) moe::cluster_sync();   // the peer's barriers exist before anyone signals them
    else __syncthreads();
    moe::tc_fence_after();
    const uint32_t tmem = S.tmem_base;
    // tiles (pair tiles when SWAP)
    const int total = WG ? p.E * wg_pair_mt(p) * p.n_tiles : S.prefix[p.E] * p.n_tiles;

    // FP8 promotion keeps 128 fp32 accumulators per epilogue thread: move
    // registers from warpgroup 0 (TMA, MMA) to the two epilogue warpgroups.
    // 128 * kRegsLow + 256 * kRegsHigh = 384 * 168, the launch allocation.
    if (warp >= 4) {
        if (FP8) moe::reg_alloc<kRegsHigh>();
        epilogue<FP8, EPI, SWAP, WG>(S, p, total, tmem, rank);
        if (!WG) zero_sentinel_rows<EPI>(p);
        if (SWAP && EPI == EPI_STORE && p.fc) fused_combine_empty_tokens(p);
    } else {
        if (FP8) moe::reg_dealloc<kRegsLow>();
        if (!SWAP && p.gx && (warp == 0 || warp - 1 < kGatherWarps) && warp != 1) {
            producer_gather<FP8, EPI>(&tmA, &tmB, stages, S, p, total, warp == 0 ? 0 : warp - 1);
            __syncwarp();
        } else if (warp == 0) {
            if (SWAP) producer_swap<EPI, WG>(&tmX, &tmB, &tmA, stages, S, p, total, rank);
            else producer<FP8, EPI>(&tmA, &tmB, stages, S, p, total);
        } else if (warp == 1) {
            if (rank == 0) mma_issuer<FP8, EPI, SWAP, WG>(stages, S, p, total, tmem);
        }
    }
    moe::tc_fence_before();
    if (SWAP) moe::cluster_sync();   // no CTA of the pair leaves while its peer may still signal it
    else __syncthreads();
    if (warp == 1) {
        moe::tc_fence_after();
        if (SWAP) moe::tmem_dealloc_pair(tmem, kTmemCols);
        else moe::tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

bool encode(CUtensorMap* map, bool fp8, const void* base, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides_bytes, const cuuint32_t* box) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint32_t estride[5] = {1, 1, 1, 1, 1};
    return fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
              static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims, strides_bytes, box, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [rows, K] (dims/strides as for encode) with boxes of 64 x 8(j + 1) rows.
bool encode_token_maps(TokenMaps* t, const void* base, const cuuint64_t* dims, const cuuint64_t* strides) {
    for (int j = 0; j < kTokenMaps; ++j) {
        const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(8 * (j + 1))};
        if (!encode(&t->m[j], false, base, 2, dims, strides, box)) return false;
    }
    return true;
}

template <bool FP8, int EPI, bool SWAP = false, bool WG = false>
moe_status_t launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const TokenMaps& tmX, const Params& p,
                    cudaStream_t s) {
    auto kern = grouped_gemm_kernel<FP8, EPI, SWAP, WG>;
    constexpr size_t kSmemBytes = smem_bytes<SWAP, EPI>();
    static int configured[64] = {0};
    int dev = 0;
    MOE_CHECK_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return MOE_ERR_CUDA;
    if (!configured[dev]) {
        MOE_CHECK_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(kSmemBytes)));
        configured[dev] = 1;
    }
    int grid = moe::sm_count();
    if (SWAP) grid &= ~1;   // whole CTA pairs
    if (grid <= 0) return MOE_ERR_CUDA;
    if (!SWAP) {
        kern<<<grid, kThreads, kSmemBytes, s>>>(tmA, tmB, tmX, p);
        MOE_CHECK_LAUNCH();
        return MOE_OK;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmX, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

// Shared by both entry points.  With gx set, A is gathered from token order
// (gx [T, K], sorted_rows [T*topk]) and the A tensor map is never used.
// The fused weighted combine of moe_grouped_gemm_combine.
struct FusedCombine {
    const int32_t* ids;
    const float* w;
    const int32_t* sorted_rows;
    const int32_t* row_pos;
    int T, k;
    int* counters;
    void* out;
};

// With weights_mn (bf16 store only) B is [E, K, N], read MN-major.  With fc
// (bf16 store only) the weighted combine is fused into the epilogue.
moe_status_t run_grouped_gemm(moe_dtype_t dtype, const void* A, const float* A_scales, const void* gx,
                              const int32_t* sorted_rows, int T, int topk, const void* B,
                              const float* B_scales, const int32_t* offsets, int E, int M_cap, int N, int K,
                              moe_epilogue_t epilogue, void* C, float* C_scales, moe_stream_t stream,
                              bool weights_mn = false, const FusedCombine* fc = nullptr) {
    MOE_CHECK_ARG(A && B && offsets && C && E >= 1 && E <= kMaxE && M_cap >= 1 && N >= 8 && K >= 8);
    MOE_CHECK_ARG(moe::aligned16(A) && moe::aligned16(B) && moe::aligned16(C));
    const bool fp8 = dtype == MOE_FP8_E4M3_B128;
    if (!fp8 && dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    const bool swiglu = epilogue == MOE_EPI_SWIGLU || epilogue == MOE_EPI_SWIGLU_QUANT_FP8;
    if (epilogue != MOE_EPI_STORE && !swiglu) return MOE_ERR_INVALID_ARG;
    if (epilogue == MOE_EPI_SWIGLU_QUANT_FP8 && !fp8) return MOE_ERR_UNSUPPORTED;
    if (swiglu) MOE_CHECK_ARG(N % 16 == 0); else MOE_CHECK_ARG(N % 8 == 0);
    if (fp8) {
        MOE_CHECK_ARG(K % 128 == 0 && A_scales && B_scales);
        // block scales are read one float at a time: a slice of a stack (an
        // expert-parallel shard) need only be 4-byte aligned
        MOE_CHECK_ARG(moe::aligned16(A_scales) && (reinterpret_cast<uintptr_t>(B_scales) & 3u) == 0);
        if (swiglu) MOE_CHECK_ARG((N / 2) % 128 == 0);
        if (epilogue == MOE_EPI_SWIGLU_QUANT_FP8) MOE_CHECK_ARG(C_scales && moe::aligned16(C_scales));
    } else {
        MOE_CHECK_ARG(K % 8 == 0);
    }
    const int esz = fp8 ? 1 : 2;
    if (gx) {
        MOE_CHECK_ARG(sorted_rows && T >= 1 && topk >= 1 && static_cast<int64_t>(T) * topk < INT_MAX);
        // gathered rows are fetched in whole 128-byte k-blocks, never past the row
        if ((static_cast<int64_t>(K) * esz) % 128 != 0) return MOE_ERR_UNSUPPORTED;
    }
    const int half = swiglu ? N / 2 : 0;
    // bf16 without a gather runs with swapped operands: weight-row tiles x
    // token tiles of up to BT rows
    const bool swap = !fp8 && !gx;
    const int feat = swap ? (swiglu ? kSwapFeatSwiglu : kSwapFeatStore) : (swiglu ? BN / 2 : BN);
    const int n_tiles = ((swiglu ? half : N) + feat - 1) / feat;
    const int64_t max_tiles = (static_cast<int64_t>(M_cap) / (swap ? BT : BM) + E) * n_tiles;
    MOE_CHECK_ARG(max_tiles < INT_MAX);
    int* err = moe::device_error_word();
    if (!err) return MOE_ERR_CUDA;

    const cuuint32_t bk = 128 / esz;  // elements in a 128-byte k-block row
    CUtensorMap tmA, tmB;
    TokenMaps tmX{};
    {
        // permuted A: 128-row tiles (swapped: token halves in boxes of 16 ..
        // 128 rows); gathered A: x [T, K] read a row at a time
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(gx ? T : M_cap)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * esz};
        const cuuint32_t box[2] = {bk, gx ? 1u : static_cast<cuuint32_t>(BM)};
        if (!swap && !encode(&tmA, fp8, A, 2, dims, strides, box)) return MOE_ERR_CUDA;
        if (swap && !encode_token_maps(&tmX, A, dims, strides)) return MOE_ERR_CUDA;
    }
    if (weights_mn) {
        if (fp8 || swiglu || gx) return MOE_ERR_UNSUPPORTED;
        // [E, K, N] with N contiguous: 64-feature x 64-row boxes (one swizzle atom)
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(E)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(N) * 2, static_cast<cuuint64_t>(K) * N * 2};
        const cuuint32_t box[3] = {64, 64, 1};
        if (!encode(&tmB, false, B, 3, dims, strides, box)) return MOE_ERR_CUDA;
        tmA = tmB;   // the M = 128 tiles load one of these boxes per CTA; tmA is only prefetched
    } else if (!swiglu) {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(E)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * esz, static_cast<cuuint64_t>(N) * K * esz};
        const cuuint32_t box[3] = {bk, swap ? 128u : BN, 1};   // swapped: 128 weight rows per CTA
        if (!encode(&tmB, fp8, B, 3, dims, strides, box)) return MOE_ERR_CUDA;
        // swapped: tmA holds the same weights in boxes of 64 rows, for the
        // M = 128 tile at the end of an expert's features
        const cuuint32_t box64[3] = {bk, 64u, 1};
        if (swap && !encode(&tmA, fp8, B, 3, dims, strides, box64)) return MOE_ERR_CUDA;
    } else if (swap) {
        // [E, N/2/8, 2, 8, K] in memory order (expert, group of 8 features,
        // gate/up, feature in group, k): one box holds 8 groups of 8 gate rows
        // and the same 8 up rows; features past N/2 are out of bounds (zeros)
        const cuuint64_t dims[5] = {static_cast<cuuint64_t>(K), 8, 2, static_cast<cuuint64_t>(half / 8),
                                    static_cast<cuuint64_t>(E)};
        const cuuint64_t strides[4] = {static_cast<cuuint64_t>(K) * esz, static_cast<cuuint64_t>(half) * K * esz,
                                       static_cast<cuuint64_t>(8) * K * esz, static_cast<cuuint64_t>(N) * K * esz};
        const cuuint32_t box[5] = {bk, 8, 2, 8, 1};
        if (!encode(&tmB, fp8, B, 5, dims, strides, box)) return MOE_ERR_CUDA;
        // tmA: 4 groups (32 features, 64 rows) per box, for the M = 128 tile
        const cuuint32_t box4[5] = {bk, 8, 2, 4, 1};
        if (!encode(&tmA, fp8, B, 5, dims, strides, box4)) return MOE_ERR_CUDA;
    } else {
        // [E, 2, N/2, K]: a gate box clips at N/2 instead of running into the up rows
        const cuuint64_t dims[4] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(half), 2,
                                    static_cast<cuuint64_t>(E)};
        const cuuint64_t strides[3] = {static_cast<cuuint64_t>(K) * esz, static_cast<cuuint64_t>(half) * K * esz,
                                       static_cast<cuuint64_t>(N) * K * esz};
        const cuuint32_t box[4] = {bk, BN / 2, 1u, 1};
        if (!encode(&tmB, fp8, B, 4, dims, strides, box)) return MOE_ERR_CUDA;
    }

    Params p;
    p.offsets = offsets;
    p.a_scales = A_scales;
    p.b_scales = B_scales;
    p.out = C;
    p.out_scales = C_scales;
    p.err = err;
    p.E = E;
    p.M_cap = M_cap;
    p.N = N;
    p.K = K;
    p.half = half;
    p.out_cols = swiglu ? half : N;
    p.n_tiles = n_tiles;
    p.k_blocks = (K + static_cast<int>(bk) - 1) / static_cast<int>(bk);
    p.nb_scale = (N + 127) / 128;
    p.gx = static_cast<const uint8_t*>(gx);
    p.sorted_rows = sorted_rows;
    p.T = gx ? T : 0;
    p.topk = gx ? topk : 1;
    p.wg_rows = 0;
    p.mn_a = weights_mn ? 1 : 0;
    p.fc = 0;
    if (fc) {
        if (fp8 || swiglu || gx || weights_mn) return MOE_ERR_UNSUPPORTED;
        p.fc = 1;
        p.ids = fc->ids;
        p.wts = fc->w;
        p.sorted_rows = fc->sorted_rows;
        p.row_pos = fc->row_pos;
        p.T = fc->T;
        p.topk = fc->k;
        p.counters = fc->counters;
        p.nfb = (N + 127) / 128;
        p.cout = fc->out;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (fp8) {
        if (epilogue == MOE_EPI_STORE) return launch<true, EPI_STORE>(tmA, tmB, tmX, p, s);
        if (epilogue == MOE_EPI_SWIGLU) return launch<true, EPI_SWIGLU>(tmA, tmB, tmX, p, s);
        return launch<true, EPI_SWIGLU_Q>(tmA, tmB, tmX, p, s);
    }
    if (swap) {
        if (epilogue == MOE_EPI_STORE) return launch<false, EPI_STORE, true>(tmA, tmB, tmX, p, s);
        return launch<false, EPI_SWIGLU, true>(tmA, tmB, tmX, p, s);
    }
    if (epilogue == MOE_EPI_STORE) return launch<false, EPI_STORE>(tmA, tmB, tmX, p, s);
    return launch<false, EPI_SWIGLU>(tmA, tmB, tmX, p, s);
}

}  // namespace

moe_status_t moe::dgrad_gemm(const void* dC, const void* B, const int32_t* offsets, int E, int M_cap, int N, int K,
                             void* dA, cudaStream_t s) {
    // dA [M_cap, K] = dC [M_cap, N] x B[e] [N, K]: a store GEMM with K output
    // features over an N-long contraction, the weights B [E, N, K] read
    // MN-major in place
    return run_grouped_gemm(MOE_BF16, dC, nullptr, nullptr, nullptr, 0, 0, B, nullptr, offsets, E, M_cap, K, N,
                            MOE_EPI_STORE, dA, nullptr, reinterpret_cast<moe_stream_t>(s), true);
}

moe_status_t moe::wgrad_gemm(const void* dC, const void* A, const void* tails, const int32_t* offsets, int E,
                             int M_cap, int N, int K, void* dB, cudaStream_t s) {
    // dB[e] [N, K] = dC_e^T A_e over expert e's rows.  Swapped operands on CTA
    // pairs: A supplies the MMA's M rows (the output features, 256 per pair
    // tile), dC its N columns (the output rows, in tiles of up to 256); both
    // are read MN-major, 64 features x 64 rows per box, from their own rows or,
    // for an expert's partial last k-block, from the zero-padded tails.
    MOE_CHECK_ARG(dC && A && tails && offsets && dB && E >= 1 && E <= kMaxE && M_cap >= 1);
    MOE_CHECK_ARG(N >= 8 && N % 8 == 0 && K >= 8 && K % 8 == 0);
    MOE_CHECK_ARG(moe::aligned16(dC) && moe::aligned16(A) && moe::aligned16(tails) && moe::aligned16(dB));
    MOE_CHECK_ARG(static_cast<int64_t>(E) * N < INT_MAX);
    const int n_tiles = (K + kSwapFeatStore - 1) / kSwapFeatStore;
    MOE_CHECK_ARG(static_cast<int64_t>(E) * ((N + BT - 1) / BT) * n_tiles < INT_MAX);
    int* err = moe::device_error_word();
    if (!err) return MOE_ERR_CUDA;
    TokenMaps tmX{};
    const cuuint32_t box[2] = {64, 64};
    const uint8_t* tail_c = static_cast<const uint8_t*>(tails);
    const uint8_t* tail_a = tail_c + static_cast<size_t>(64) * E * N * 2;
    const struct { const void* base; int cols; cuuint64_t rows; } ops[4] = {
        {A, K, static_cast<cuuint64_t>(M_cap)}, {dC, N, static_cast<cuuint64_t>(M_cap)},
        {tail_a, K, static_cast<cuuint64_t>(64) * E}, {tail_c, N, static_cast<cuuint64_t>(64) * E}};
    for (int i = 0; i < kWgMaps; ++i) {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(ops[i].cols), ops[i].rows};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ops[i].cols) * 2};
        if (!encode(&tmX.m[i], false, ops[i].base, 2, dims, strides, box)) return MOE_ERR_CUDA;
    }
    Params p{};
    p.offsets = offsets;
    p.out = dB;
    p.err = err;
    p.E = E;
    p.M_cap = M_cap;
    p.N = K;
    p.K = 64;
    p.half = 0;
    p.out_cols = K;
    p.n_tiles = n_tiles;
    p.k_blocks = 0;
    p.nb_scale = 0;
    p.topk = 1;
    p.wg_rows = N;
    return launch<false, EPI_STORE, true, true>(tmX.m[kWgA], tmX.m[kWgC], tmX, p, s);
}

extern "C" moe_status_t moe_grouped_gemm(moe_dtype_t dtype, const void* A, const float* A_scales,
                                         const void* B, const float* B_scales, const int32_t* offsets,
                                         int E, int M_cap, int N, int K, moe_epilogue_t epilogue,
                                         void* C, float* C_scales, moe_stream_t stream) {
    return run_grouped_gemm(dtype, A, A_scales, nullptr, nullptr, 0, 0, B, B_scales, offsets, E, M_cap, N, K,
                            epilogue, C, C_scales, stream);
}

extern "C" size_t moe_grouped_gemm_combine_workspace_size(int T, int H) {
    if (T < 1 || H < 8) return 0;
    const size_t bytes = static_cast<size_t>(T) * ((H + 127) / 128) * sizeof(int);
    return (bytes + 255) & ~static_cast<size_t>(255);
}

extern "C" moe_status_t moe_grouped_gemm_combine(const void* h, const void* W2, const int32_t* offsets, int E,
                                                 int M_cap, int H, int I, const int32_t* topk_ids,
                                                 const float* topk_w, const int32_t* sorted_rows,
                                                 const int32_t* row_pos, int T, int k, void* Y2, void* out,
                                                 void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_CHECK_ARG(topk_ids && topk_w && sorted_rows && row_pos && out && T >= 1 && k >= 1 && k <= 32);
    MOE_CHECK_ARG(static_cast<int64_t>(T) * k <= M_cap && H % 8 == 0);
    MOE_CHECK_ARG(moe::aligned16(out) && moe::aligned16(topk_ids) && moe::aligned16(topk_w));
    const size_t need = moe_grouped_gemm_combine_workspace_size(T, H);
    if (!ws || ws_bytes < need) return MOE_ERR_WORKSPACE;
    MOE_CHECK_ARG(moe::aligned16(ws));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    MOE_CHECK_CUDA(cudaMemsetAsync(ws, 0, need, s));   // the per-(token, block) counters
    const FusedCombine fc{topk_ids, topk_w, sorted_rows, row_pos, T, k, static_cast<int*>(ws), out};
    return run_grouped_gemm(MOE_BF16, h, nullptr, nullptr, nullptr, 0, 0, W2, nullptr, offsets, E, M_cap, H, I,
                            MOE_EPI_STORE, Y2, nullptr, stream, false, &fc);
}

extern "C" moe_status_t moe_grouped_gemm_gather(moe_dtype_t dtype, const void* x, const float* x_scales, int T,
                                                int k, const int32_t* sorted_rows, const void* B,
                                                const float* B_scales, const int32_t* offsets, int E, int M_cap,
                                                int N, int K, moe_epilogue_t epilogue, void* C, float* C_scales,
                                                moe_stream_t stream) {
    MOE_CHECK_ARG(x && sorted_rows);
    return run_grouped_gemm(dtype, x, x_scales, x, sorted_rows, T, k, B, B_scales, offsets, E, M_cap, N, K,
                            epilogue, C, C_scales, stream);
}
