// Tensor-core GEMMs of the TP-MLP block on sm_103a: TMA -> shared memory ring ->
// tcgen05.mma (one thread) -> fp32 accumulators in tensor memory -> epilogue
// warps (tcgen05.ld) -> fused bias / GeLU / GeLU' / shard fold -> global memory.
//
// Tiles are 256 x 256 on CTA pairs (a 2-CTA cluster, tcgen05 cta_group::2: each
// CTA loads its 128 rows of A and 128 of B's 256 columns, the even CTA issues the
// MMAs, each CTA's TMEM holds its 128 rows of the accumulator) or 128 x 256 on
// single CTAs.  Outputs at most 128 wide take 256 x 128 tiles on CTA pairs.  The
// plain-store and GeLU epilogues (no shard fold) can take 256 x 512 tiles on CTA
// pairs instead: two MMAs of N = 256 per k-step into the two halves of the 512
// TMEM columns, which loads a quarter fewer operand bytes per FLOP (see Cfg).
// One persistent CTA per SM, 10 warps:
//   warp 0      TMA producer (one elected lane): fills a ring of stages (4 to 8)
//               of 128x64 A tiles and B tiles of the CTA's columns, 128-byte
//               swizzled.
//   warp 1      MMA issuer (one elected lane) and owner of the 512 TMEM columns:
//               two fp32 accumulators (128 lanes x tile width), used alternately
//               per "accumulation unit" (one K range of one output tile).
//   warps 2..9  epilogue: warp w reads TMEM lanes 32*(w%4)..+31 (its rows) and
//               one half of the accumulator's columns, (w-2)/4.
//
// The all-reduce of the t shard partials ("Megatron-LM" report, section 4.1,
// Z = sum_i Y_i B_i; section 4.2 for dX in the backward direction) becomes the
// FOLD epilogues: each shard's K range is its own accumulation unit, so each
// partial Z_i is a complete fp32 product in TMEM; the epilogue threads pull it
// into registers and add it to their running sum in the order the shards come,
// ((Z_1 + Z_2) + Z_3) + ... (descending, ((Z_t + Z_t-1) + ...), for the tiles of
// odd waves, which walk K downwards), releasing the TMEM buffer at once so the
// tensor core starts the next shard in the other buffer without waiting.
//
// Every wait is bounded (mbar_wait); a wait that runs out records
// TPMLP_ERR_TIMEOUT in the status word, raises a CTA-wide abort flag, and the CTA
// drains its own copies and MMAs and frees its tensor memory before returning.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace tpmlp {
namespace tc {

constexpr int BM = 128;   // accumulator rows per CTA (TMEM lanes)
constexpr int BN = 256;   // accumulator columns of the wide tile (the narrow one has 128)
constexpr int BK = 64;    // 64 bf16 = one 128-byte swizzle row
constexpr int NUM_THREADS = 320;
constexpr int EPI_THREADS = 256;
constexpr uint32_t TMEM_COLS = 512;
constexpr int MN_BLOCK_BYTES = 64 * BK * 2;             // one 64(MN) x 64(K) TMA box
// Epilogue staging: each epilogue warp owns two 32 x 32 bf16 boxes (2 KB each,
// 64-byte swizzled) that it fills from registers and writes out with TMA stores.
// The dS epilogue owns two 32 x 64 bf16 boxes (4 KB each, 128-byte swizzled):
// one for the dS it stores, one for the P it loads.
constexpr int STG_BOX = 32 * 32 * 2;
constexpr int STG_BOX_WIDE = 32 * 64 * 2;

// Per-CTA pipeline geometry.  CG = 1: one CTA computes a 128 x 256 tile and loads
// all of B's 256 columns.  CG = 2: a CTA pair computes a 256 x 256 tile with
// CTA-pair MMAs; each CTA loads its own 128 rows of A and 128 of B's columns, so
// a stage is 32 KB instead of 48 KB and six stages fit.
//
// TILE_N = 128 (CTA pairs only) is the narrow tile for outputs at most 128 wide
// (the per-head products with N = d): each CTA loads 64 of B's columns, a stage
// is 24 KB and eight stages fit.
//
// TILE_N = 512 (CTA pairs only) is the wide tile: each CTA loads 128 rows of A
// and 256 of B's columns (a 48 KB stage, four of them), and one k-step is two
// MMAs of 256 x 256 x 16, one per half of the tile's columns, into the two
// 256-column halves of the CTA's TMEM.  Per SM that is 48 KB of operands per
// 8.4 MFLOP instead of 32 KB per 4.2 MFLOP: 25% fewer bytes from L2 per FLOP,
// and 15% less shared-memory traffic (TMA writes plus MMA reads) per FLOP.
// The accumulator is no longer double-buffered; the MMA warp starts a tile's
// first half as soon as the epilogue has drained that half of the previous
// tile (see the MMA issuer).
template <int CG, int TILE_N_ = BN, int EPI_ = EPI_STORE>
struct Cfg {
    static constexpr int TILE_M = BM * CG;
    static constexpr int TILE_N = TILE_N_;
    static constexpr int B_ROWS = TILE_N / CG;
    static constexpr int A_STAGE = BM * BK * 2;
    static constexpr int B_STAGE = B_ROWS * BK * 2;
    static constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
    static constexpr bool DS = EPI_ == EPI_ATTN_DS;
    static constexpr int STG_PER_WARP = DS ? 2 * STG_BOX_WIDE : 2 * STG_BOX;
    // dS: the K extent is one head dimension (two K blocks per tile), so fewer
    // stages make room for its wider staging boxes
    static constexpr int STAGES = CG == 1 ? (DS ? 3 : 4) : (TILE_N == BN ? (DS ? 5 : 6) : (TILE_N == 512 ? 4 : 8));
    static constexpr int SMEM_DYN = STAGES * STAGE_BYTES + (EPI_THREADS / 32) * STG_PER_WARP + 1024;
};
constexpr int MAX_STAGES = 8;

constexpr uint32_t STATUS_TIMEOUT = 4;  // TPMLP_ERR_TIMEOUT
constexpr uint32_t STATUS_DEVICE = 5;   // TPMLP_ERR_DEVICE: a bounds check of the TPMLP_DEBUG build failed

// The TPMLP_DEBUG build (libtpmlp_debug.so) checks, before every TMA copy, MMA,
// TMEM load and global store of the kernel, that the tile coordinates, k-block
// range, shared-memory addresses, TMEM columns and partial-sum indices lie inside
// what the launch set up.  A failed check records TPMLP_ERR_DEVICE and the check's
// code in the status word, raises the CTA's abort flag and skips the access; the
// kernel then winds down like after a timeout.  It stands in for a memory checker
// on a machine where none can run.  In the normal build every check is a
// constant true and compiles away.
#ifndef TPMLP_DEBUG
#define TPMLP_DEBUG 0
#endif

struct Params {
    int M, N;
    int m_tiles, n_tiles;
    int group;     // tiles walk `group` M-tiles (or N-tiles if raster_n) fastest
    int raster_n;  // 0: groups along M; 1: groups along N
    int nshards, kb_per_shard;
    void *out0;
    void *out1;
    const void *aux;
    const void *bias;
    uint32_t *status;
    unsigned long long wait_ns;
    float *colsum_part;  // GeLU' epilogue: fp32 column sums of dY per 32-row block, or null
    int batch;           // independent problems, tiles of problem z follow those of z - 1
    float scale;
    int causal;
    const float *rowvec;
    int causal_k;    // K range of an M-tile: 0 all; 1 k < end of the tile's rows; 2 k >= start of its rows
    int skip_upper;  // tiles wholly above the diagonal (every column past every row) are not computed
    int flip_odd;    // odd problems walk their M-tiles in reverse order (load balance under causal ranges)
    // Causal K ranges over one column of tiles: each unit takes the M-tiles of
    // a problem in complementary pairs (see tile_coords); `units` is the grid's
    // unit count, which the pair order is laid out for.
    int pair_order;
    int units;
    int a_mn4, b_mn4;  // MN-major operand mapped as 4-D (all of a stage's 64-wide blocks in one copy)
    // Bias gradient from the MMA (EPI_STORE with MN-major A): one extra M-tile
    // whose A is a 64 x 64 block of ones (map tmO2), so its first accumulator
    // row is 1^T B, the column sums of the B operand over K; written to bias_grad.
    int bias_tile;
    void *bias_grad;
    // Per-head problems read and written in place in token-major arrays (kernels
    // instantiated with HEADS): the rank of each operand's and the output's map.
    // Rank 3: (x, y, z); rank 4: (x, y, g, b); rank 5: (x, y, j, i, b), where
    // problem z = b * heads + g and head g = i * hpt + j (hpt heads per shard).
    int a_rank, b_rank, o_rank;
    int heads, hpt;
    // Wide tiles (TILE_N = 512): the last `wide_tail` tiles of the order are each
    // split into their two 256-column halves, run as separate half-width tiles,
    // so that a last partial wave of wide tiles is spread over twice the units.
    int wide_tail;
    // Wide tiles: the tiles of every odd wave (slot / units odd) walk K from the
    // last k-block down to the first, so that a unit's next tile starts on the
    // k-blocks its wave read last, while they are still in L2.
    int serpentine;
};

// Coordinates after (x, y) of problem z in a map of the given rank.
__device__ __forceinline__ void head_coords(int rank, int z, int heads, int hpt, int &c2, int &c3, int &c4) {
    if (rank <= 3) {
        c2 = z, c3 = 0, c4 = 0;
        return;
    }
    const int g = z % heads, b = z / heads;
    if (rank == 4)
        c2 = g, c3 = b, c4 = 0;
    else
        c2 = g % hpt, c3 = g / hpt, c4 = b;
}

template <bool PAIR>
__device__ __forceinline__ void tma_load_rank(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x, int y,
                                              int rank, int c2, int c3, int c4) {
    if (rank <= 3) {
        if constexpr (PAIR)
            ptx::tma_load_3d_pair(dst, map, bar, x, y, c2);
        else
            ptx::tma_load_3d(dst, map, bar, x, y, c2);
    } else if (rank == 4) {
        if constexpr (PAIR)
            ptx::tma_load_4d_pair(dst, map, bar, x, y, c2, c3);
        else
            ptx::tma_load_4d(dst, map, bar, x, y, c2, c3);
    } else {
        if constexpr (PAIR)
            ptx::tma_load_5d_pair(dst, map, bar, x, y, c2, c3, c4);
        else
            ptx::tma_load_5d(dst, map, bar, x, y, c2, c3, c4);
    }
}

__device__ __forceinline__ void tma_store_rank(const CUtensorMap *map, uint32_t src, int x, int y, int rank, int c2,
                                               int c3, int c4) {
    if (rank <= 3)
        ptx::tma_store_3d(map, src, x, y, c2);
    else if (rank == 4)
        ptx::tma_store_4d(map, src, x, y, c2, c3);
    else
        ptx::tma_store_5d(map, src, x, y, c2, c3, c4);
}

// Causal per-head products.  Square per-head problems (M = K = seq) whose A or B
// operand is zero above the diagonal need only part of K: P V and dS K only keys
// up to the tile's last query (causal_k = 1), P^T dO and dS^T Q only queries from
// the tile's first key on (causal_k = 2).  The range ends are multiples of the
// tile height, so of BK.  With nshards = 1 the range is [kb0, kb1) in k-blocks.
template <int TILE_M>
__device__ __forceinline__ void k_range(const Params &p, int mb, int &kb0, int &kb1) {
    kb0 = 0;
    kb1 = p.nshards * p.kb_per_shard;
    if (p.causal_k == 1) kb1 = min(kb1, (mb + 1) * (TILE_M / BK));
    else if (p.causal_k == 2) kb0 = mb * (TILE_M / BK);
}

// Scores and dS are not needed above the diagonal: a tile whose first column lies
// past its last row is skipped by every role (none of its outputs is read).
template <int TILE_M, int TILE_N = BN>
__device__ __forceinline__ bool tile_active(const Params &p, int mb, int nb) {
    return !p.skip_upper || nb * TILE_N <= mb * TILE_M + TILE_M - 1;
}

// Tile order: super-rows of `group` tiles along one dimension; inside a
// super-row the grouped index runs fastest, so the CTAs resident at one time
// share `group` panels of one operand and a few of the other.
__device__ __forceinline__ void tile_coords(int tile, const Params &p, int &mb, int &nb, int &zb) {
    if (p.pair_order) {
        // Causal K ranges with one N-tile per problem (the products against P or
        // dS, N = d): M-tile i of a problem costs i + 1 k-blocks of 256 keys, or
        // m_tiles - i, so M-tiles i and m_tiles - 1 - i together cost the same
        // for every i.  The slots of unit u are u, u + U, u + 2U, ... (U units);
        // slots 2jU + u and (2j + 1)U + u hold the two M-tiles of pair jU + u,
        // so every unit runs whole pairs of equal cost.  The R = n / 2U full
        // double rounds are laid out this way; of the s = n - 2RU slots left,
        // units that get two take one more pair, the others one tile each.
        const int U = p.units, half = p.m_tiles >> 1;
        const int n = p.m_tiles * p.batch;
        const int R = n / (2 * U), s = n - 2 * R * U;
        const int k = tile / U, u = tile - k * U;
        const int twice = s > U ? s - U : 0;  // units with two slots left
        int pair, member;
        if (k < 2 * R) {
            pair = u + (k >> 1) * U;
            member = k & 1;
        } else if (u < twice) {
            pair = R * U + u;
            member = k - 2 * R;
        } else {
            const int v = u - twice;
            pair = R * U + twice + (v >> 1);
            member = v & 1;
        }
        zb = pair / half;
        const int i = pair - zb * half;
        mb = member ? i : p.m_tiles - 1 - i;
        nb = 0;
        return;
    }
    const int per_batch = p.m_tiles * p.n_tiles;
    zb = tile / per_batch;
    tile -= zb * per_batch;
    const int fast_tiles = p.raster_n ? p.n_tiles : p.m_tiles;
    const int slow_tiles = p.raster_n ? p.m_tiles : p.n_tiles;
    const int per_group = p.group * slow_tiles;
    const int g = tile / per_group;
    const int first = g * p.group;
    const int gsize = min(fast_tiles - first, p.group);
    const int local = tile - g * per_group;
    const int fast = first + local % gsize;
    const int slow = local / gsize;
    mb = p.raster_n ? slow : fast;
    nb = p.raster_n ? fast : slow;
    // Under causal K ranges (or skipped upper tiles) an M-tile's work grows or
    // shrinks with its index.  A unit takes every num_units-th tile, so problems
    // walked in order hand each unit the same few M-tile indices again and again
    // (76 units and 8 M-tiles: two indices per unit).  Walking the M-tiles of
    // every odd problem backwards gives each unit a mix of heavy and light
    // tiles, and the tiles of one problem stay adjacent (sharing operands in L2).
    if (p.flip_odd && (zb & 1)) mb = p.m_tiles - 1 - mb;
}

// Wide tiles: the tile order is that of tile_coords over the 256 x 512 tiles,
// except that each of the last p.wide_tail of them is run as two half-width
// tiles.  hm is the set of column halves the slot covers: 3 both, 1 the first
// 256-column half (TMEM columns 0..255), 2 the second (TMEM columns 256..511).
__device__ __forceinline__ void wide_coords(int tile, const Params &p, int &mb, int &nb, int &zb, int &hm) {
    const int full = p.m_tiles * p.n_tiles * p.batch - p.wide_tail;
    int wt = tile;
    hm = 3;
    if (tile >= full) {
        const int j = tile - full;
        wt = full + (j >> 1);
        hm = 1 << (j & 1);
    }
    tile_coords(wt, p, mb, nb, zb);
}

// Records a timeout once in the status word (detail = which role gave up).
__device__ __forceinline__ void record_timeout(const Params &p, volatile int *abort_flag,
                                               uint32_t role) {
    *abort_flag = 1;
    if (p.status) {
        if (atomicCAS(p.status, 0u, STATUS_TIMEOUT) == 0u) atomicExch(p.status + 1, role);
    }
}

// Debug-build bounds check (see TPMLP_DEBUG above): true if `cond` holds.
// code = (check << 8) | role, role 1 producer, 2 MMA issuer, 3 epilogue.
__device__ __forceinline__ bool dbg_ok(bool cond, const Params &p, volatile int *abort_flag, uint32_t code) {
#if TPMLP_DEBUG
    if (!cond) {
        *abort_flag = 1;
        if (p.status && atomicCAS(p.status, 0u, STATUS_DEVICE) == 0u) atomicExch(p.status + 1, code);
    }
    return cond;
#else
    (void)cond, (void)p, (void)abort_flag, (void)code;
    return true;
#endif
}

__device__ __forceinline__ uint32_t dynamic_smem_bytes() {
    uint32_t n;
    asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(n));
    return n;
}

// The tanh form of GeLU, with c = sqrt(2/pi) and k = 0.044715:
//   GeLU(x)  = x/2 (1 + tanh u),  u = c (x + k x^3) = x (c + c k x^2)
//   GeLU'(x) = (1 + tanh u)/2 + (1 - tanh^2 u) x/2 (c + 3 c k x^2)
// with the constant products folded, so that each costs a handful of FMAs
// around the one tanh.
constexpr float kGeluC = 0.7978845608028654f;           // c
constexpr float kGeluCK = 0.035677408136300125f;        // c k
constexpr float kGeluHalfC = 0.3989422804014327f;       // c / 2
constexpr float kGeluThreeHalfCK = 0.05351611220445019f;  // 3 c k / 2

__device__ __forceinline__ float gelu_f(float x) {
    const float u = x * fmaf(kGeluCK, x * x, kGeluC);
    const float hx = 0.5f * x;
    return fmaf(hx, ptx::tanh_approx(u), hx);
}

__device__ __forceinline__ float gelu_prime_f(float x) {
    const float x2 = x * x;
    const float th = ptx::tanh_approx(x * fmaf(kGeluCK, x2, kGeluC));
    const float hxdu = x * fmaf(kGeluThreeHalfCK, x2, kGeluHalfC);  // x/2 du/dx
    return fmaf(fmaf(-th, th, 1.0f), hxdu, fmaf(0.5f, th, 0.5f));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void unpack_bf16(uint32_t u, float &lo, float &hi) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&u);
    lo = __low2float(v);
    hi = __high2float(v);
}

// Stores 8 consecutive fp32 values as bf16 at out[off .. off+7] (16 bytes).
__device__ __forceinline__ void store8(void *out, int64_t off, const float *v) {
    uint4 w;
    w.x = pack_bf16(v[0], v[1]);
    w.y = pack_bf16(v[2], v[3]);
    w.z = pack_bf16(v[4], v[5]);
    w.w = pack_bf16(v[6], v[7]);
    *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(out) + off) = w;
}

__device__ __forceinline__ void load8(const void *in, int64_t off, float *v) {
    const uint4 w = __ldg(reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(in) + off));
    unpack_bf16(w.x, v[0], v[1]);
    unpack_bf16(w.y, v[2], v[3]);
    unpack_bf16(w.z, v[4], v[5]);
    unpack_bf16(w.w, v[6], v[7]);
}

// 32 consecutive bf16 bias values fetched ahead of the chunk that adds them, so
// that the load's latency overlaps the work before it.  Values past N read as
// zero (the bias is a row-major vector of N bf16).
struct BiasPre {
    uint4 w[4];
};
__device__ __forceinline__ void bias_fetch(const void *bias, int col, int N, BiasPre &b) {
    const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(bias) + col);
#pragma unroll
    for (int g = 0; g < 4; ++g) b.w[g] = col + 8 * g < N ? __ldg(src + g) : make_uint4(0u, 0u, 0u, 0u);
}
__device__ __forceinline__ void bias_unpack(const BiasPre &b, float (&v)[32]) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        unpack_bf16(b.w[g].x, v[8 * g], v[8 * g + 1]);
        unpack_bf16(b.w[g].y, v[8 * g + 2], v[8 * g + 3]);
        unpack_bf16(b.w[g].z, v[8 * g + 4], v[8 * g + 5]);
        unpack_bf16(b.w[g].w, v[8 * g + 6], v[8 * g + 7]);
    }
}

// Row r of a 32 x 32 bf16 box staged for a 64-byte-swizzled TMA store: 16-byte
// chunk j of the 64-byte row sits at chunk j ^ ((r >> 1) & 3).
__device__ __forceinline__ void stage_row(uint32_t box, int r, const uint32_t (&w)[16]) {
    const uint32_t row = box + static_cast<uint32_t>(r) * 64u;
    const int x = (r >> 1) & 3;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        ptx::st_shared_v4(row + (static_cast<uint32_t>(j ^ x) << 4), w[4 * j], w[4 * j + 1], w[4 * j + 2],
                          w[4 * j + 3]);
}

// Reads row r of a 64-byte-swizzled 32 x 32 bf16 box (the layout a TMA load
// with SWIZZLE_64B leaves) as 32 floats.
__device__ __forceinline__ void unstage_row(uint32_t box, int r, float (&v)[32]) {
    const uint32_t row = box + static_cast<uint32_t>(r) * 64u;
    const int x = (r >> 1) & 3;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t w[4];
        ptx::ld_shared_v4(row + (static_cast<uint32_t>(j ^ x) << 4), w[0], w[1], w[2], w[3]);
#pragma unroll
        for (int i = 0; i < 4; ++i) unpack_bf16(w[i], v[8 * j + 2 * i], v[8 * j + 2 * i + 1]);
    }
}

// Column half hf (32 of the 64 bf16 columns) of row r of a 32 x 64 bf16 box in
// the 128-byte-swizzled layout: 16-byte chunk j of the 128-byte row sits at
// chunk j ^ (r & 7).  stage_half_row128 fills it for a TMA store;
// unstage_half_row128 reads what a TMA load with SWIZZLE_128B left.
__device__ __forceinline__ void stage_half_row128(uint32_t box, int r, int hf, const uint32_t (&w)[16]) {
    const uint32_t row = box + static_cast<uint32_t>(r) * 128u;
    const int x = r & 7;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        ptx::st_shared_v4(row + (static_cast<uint32_t>((4 * hf + j) ^ x) << 4), w[4 * j], w[4 * j + 1],
                          w[4 * j + 2], w[4 * j + 3]);
}
__device__ __forceinline__ void unstage_half_row128(uint32_t box, int r, int hf, float (&v)[32]) {
    const uint32_t row = box + static_cast<uint32_t>(r) * 128u;
    const int x = r & 7;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t w[4];
        ptx::ld_shared_v4(row + (static_cast<uint32_t>((4 * hf + j) ^ x) << 4), w[0], w[1], w[2], w[3]);
#pragma unroll
        for (int i = 0; i < 4; ++i) unpack_bf16(w[i], v[8 * j + 2 * i], v[8 * j + 2 * i + 1]);
    }
}

__device__ __forceinline__ void pack32(const float (&v)[32], uint32_t (&w)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack_bf16(v[2 * i], v[2 * i + 1]);
}

// Loads 32 consecutive bf16 values of a row-major [rows, N] matrix; entries past
// the end of the row (ragged N) or of the matrix (ok = false) read as zero.
__device__ __forceinline__ void load32(const void *in, int64_t off, int col, int N, bool ok, float (&v)[32]) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        if (ok && col + 8 * g < N) {
            load8(in, off + 8 * g, &v[8 * g]);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[8 * g + i] = 0.0f;
        }
    }
}

// Column sums of the warp's staged 32 x 32 bf16 box (64-byte swizzle, row r at
// byte 64 r, 16-byte chunk j of the row at chunk j ^ ((r >> 1) & 3)).  Lane l
// adds the bf16 pair in word l & 15 of its rows over one half of the box, rows
// 16 (l >> 4) .. +15 in order, the upper half taking the rows of each pair
// swapped so that the two halves read disjoint banks.  One exchange then adds
// the two halves' sums: lane l returns the sum over all 32 rows of column
// 2 (l & 15) + (l >> 4).  The summation order is the same on every run.
__device__ __forceinline__ float box_colsum32(uint32_t box, int lane) {
    const int w = lane & 15, hi = lane >> 4;
    float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int r = 16 * hi + (i ^ hi);
        const int chunk = (w >> 2) ^ ((i >> 1) & 3);  // (r >> 1) & 3 == (i >> 1) & 3
        const uint32_t addr = box + static_cast<uint32_t>(r) * 64u + (static_cast<uint32_t>(chunk) << 4) +
                              (static_cast<uint32_t>(w & 3) << 2);
        float lo, up;
        unpack_bf16(ptx::ld_shared_u32(addr), lo, up);
        s0 += lo;
        s1 += up;
    }
    const float send = hi ? s0 : s1;
    const float keep = hi ? s1 : s0;
    return keep + __shfl_xor_sync(0xffffffffu, send, 16);
}

// Finishes one 32-column chunk of this thread's row: applies the epilogue
// operation to the fp32 accumulator values and writes the result (two results
// for bias + GeLU) through the warp's staging boxes with TMA stores.  Rows and
// columns outside the output are clipped by the TMA unit.
// The GeLU' epilogue reads H through the warp's second staging box: a TMA load
// of the 32 x 32 H chunk is kept one chunk ahead of the chunk being finished.
struct AuxLoad {
    uint32_t bar;    // this warp's barrier
    uint32_t phase;  // parity of the next completion
    bool pending;    // a load has been issued and not yet consumed
};

__device__ __forceinline__ void aux_issue(const CUtensorMap *tm, AuxLoad &a, uint32_t box, int col, int row0,
                                          int z, int lane, uint32_t bytes = STG_BOX) {
    __syncwarp();  // every lane has read the previous chunk out of the box
    if (lane == 0) {
        ptx::bulk_wait_read0();  // a store staged in this box (rebuilt Y) or the previous one has been read
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive_expect_tx(a.bar, bytes);
        ptx::tma_load_3d(box, tm, a.bar, col, row0, z);  // out-of-range parts read as zero
    }
    a.pending = true;
}

// 32 consecutive column sums (fp32) to the bf16 bias gradient, past N skipped.
__device__ __forceinline__ void store_bias_grad(const Params &p, int col, const float (&v)[32]) {
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.bias_grad);
#pragma unroll
    for (int i = 0; i < 32; ++i)
        if (col + i < p.N) out[col + i] = __float2bfloat16_rn(v[i]);
}

// y = GeLU(h) for 32 bf16 values packed in pairs (fp32 arithmetic, bf16 result).
__device__ __forceinline__ void gelu_of_packed(const uint32_t (&h)[16], uint32_t (&y)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float a, b;
        unpack_bf16(h[i], a, b);
        y[i] = pack_bf16(gelu_f(a), gelu_f(b));
    }
}

template <int EPI, bool HEADS = false>
__device__ __forceinline__ void finish_chunk(const Params &p, const CUtensorMap *tm0, const CUtensorMap *tm1,
                                             const CUtensorMap *tm2, float (&v)[32], int64_t row, int row0,
                                             int col, int z, int lane, uint32_t stg, AuxLoad *aux = nullptr,
                                             int next_col = -1, int next_row0 = 0,
                                             volatile int *abort_flag = nullptr,
                                             const BiasPre *bias_pre = nullptr) {
    if constexpr (EPI == EPI_ATTN_SCORE) {
        // S = scale * Q K^T with the causal mask, stored in fp16 for the softmax
        // (11 significant bits; finite values saturate at the fp16 range, the
        // masked ones are -inf).  Only a chunk that reaches past the diagonal
        // (its last column beyond its first row) has masked entries.
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = ptx::f16x2_satfinite(v[2 * i] * p.scale, v[2 * i + 1] * p.scale);
        if (p.causal && col + 31 > row0) {
            constexpr uint32_t NEG_INF_LO = 0x0000FC00u, NEG_INF_HI = 0xFC000000u;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if (col + 2 * i > row) w[i] = NEG_INF_HI | NEG_INF_LO;
                else if (col + 2 * i + 1 > row) w[i] = (w[i] & 0x0000FFFFu) | NEG_INF_HI;
            }
        }
        if (lane == 0) ptx::bulk_wait_read0();
        __syncwarp();
        stage_row(stg, lane, w);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && row0 < p.M && col < p.N) {
            ptx::tma_store_3d(tm0, stg, col, row0, z);
            ptx::bulk_commit();
        }
        return;
    }
    uint32_t w0[16], w1[16];
    bool two = false, store0 = true;
    const CUtensorMap *tm_second = tm1;  // map of the second staged box
    if constexpr (EPI == EPI_BIAS_GELU) {
        // out0 = acc + bias (unless null); out1 = GeLU of it, or with out1 null
        // no activation at all (a plain biased projection)
        // Y is GeLU of H as stored (rounded to bf16), the same value the
        // backward's recomputation rebuilds from the saved H.
        float bias[32];
        if (bias_pre != nullptr)
            bias_unpack(*bias_pre, bias);
        else
            load32(p.bias, col, col, p.N, true, bias);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] += bias[i];
        pack32(v, w0);
        if (p.out1 != nullptr) {
            gelu_of_packed(w0, w1);
            two = true;
        }
        store0 = p.out0 != nullptr;
    } else if constexpr (EPI == EPI_DGELU) {
        float hv[32];
        bool got = ptx::mbar_wait(aux->bar, aux->phase, p.wait_ns, abort_flag);
        aux->phase ^= 1u;
        aux->pending = false;
        if (!__all_sync(0xffffffffu, got)) {
            if (lane == 0) record_timeout(p, abort_flag, 6);
        }
        unstage_row(stg + STG_BOX, lane, hv);
        // With activation recomputation the H box is reused to stage the rebuilt
        // Y, so the next H load waits until that store has left the box.
        const bool rebuild_y = p.out1 != nullptr;
        if (!rebuild_y && next_col >= 0) aux_issue(tm1, *aux, stg + STG_BOX, next_col, next_row0, z, lane);
        if (rebuild_y) {
            float y[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) y[i] = gelu_f(hv[i]);
            pack32(y, w1);
            two = true;
            tm_second = tm2;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= gelu_prime_f(hv[i]);
        pack32(v, w0);
    } else if constexpr (EPI == EPI_FOLD_BIAS) {
        float bias[32];
        load32(p.bias, col, col, p.N, true, bias);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] += bias[i];
        pack32(v, w0);
    } else {  // EPI_STORE, EPI_FOLD
        pack32(v, w0);
    }
    // The previous chunk's stores must have finished reading the staging boxes.
    if (lane == 0) ptx::bulk_wait_read0();
    __syncwarp();
    stage_row(stg, lane, w0);
    if (two) stage_row(stg + STG_BOX, lane, w1);
    ptx::fence_proxy_async_smem();
    __syncwarp();
    // A box that lies wholly outside the output (ragged last tile) is not stored.
    if (lane == 0 && row0 < p.M && col < p.N) {
        if (store0) {
            if constexpr (HEADS) {
                int c2, c3, c4;
                head_coords(p.o_rank, z, p.heads, p.hpt, c2, c3, c4);
                tma_store_rank(tm0, stg, col, row0, p.o_rank, c2, c3, c4);
            } else {
                ptx::tma_store_3d(tm0, stg, col, row0, z);
            }
        }
        if (two) ptx::tma_store_3d(tm_second, stg + STG_BOX, col, row0, z);
        ptx::bulk_commit();
    }
    if constexpr (EPI == EPI_DGELU) {
        if (p.colsum_part) {
            // da = 1^T dY: column sums of the stored (bf16-rounded) dY of this
            // warp's 32 rows, read back from the staged box (the TMA store only
            // reads it too).  Rows past M hold exact zeros (zero-filled operands).
            const float cs = box_colsum32(stg, lane);
            const int c = col + 2 * (lane & 15) + (lane >> 4);
            if (row0 < p.M && c < p.N) p.colsum_part[static_cast<int64_t>(row0 >> 5) * p.N + c] = cs;
        }
        if (p.out1 != nullptr && next_col >= 0) aux_issue(tm1, *aux, stg + STG_BOX, next_col, next_row0, z, lane);
    }
}

// dS = P * (dP - D) * scale for column half hf of a 64-column pair of chunks:
// P comes from the warp's P box (128-byte rows, loaded by TMA), D is one fp32
// per row, and the result is staged in the same half of the store box.
__device__ __forceinline__ void ds_half(const Params &p, float (&v)[32], int64_t row, int z, int lane,
                                        uint32_t sbox, uint32_t pbox, int hf) {
    float pv[32];
    unstage_half_row128(pbox, lane, hf, pv);
    const float D = row < p.M ? p.rowvec[static_cast<int64_t>(z) * p.M + row] : 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = pv[i] * (v[i] - D) * p.scale;
    uint32_t w[16];
    pack32(v, w);
    stage_half_row128(sbox, lane, hf, w);
}

template <int EPI, bool A_MN, bool B_MN, int CG, bool HEADS, int TILE_N>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmO0, const __grid_constant__ CUtensorMap tmO1,
                const __grid_constant__ CUtensorMap tmO2, const __grid_constant__ CUtensorMap tmB2,
                const Params p) {
    using C = Cfg<CG, TILE_N, EPI>;
    constexpr bool PAIR = CG == 2;
    constexpr bool FOLD = (EPI == EPI_FOLD_BIAS || EPI == EPI_FOLD);
    constexpr bool WIDE = TILE_N == 512;
    constexpr int MMA_N = WIDE ? 256 : TILE_N;  // N of one MMA instruction
    constexpr uint32_t IDESC = ptx::idesc_bf16_f32(C::TILE_M, MMA_N, A_MN, B_MN);
    // each epilogue warp finishes TILE_N / 2 columns of its 32 rows, in 32-column chunks
    constexpr int CHUNKS = TILE_N / 64;
    static_assert(TILE_N == BN || TILE_N == 512 || (TILE_N == 128 && CG == 2 && EPI == EPI_STORE),
                  "narrow tile: CTA pairs, plain store");
    static_assert(!WIDE || (CG == 2 && !HEADS && (EPI == EPI_STORE || EPI == EPI_BIAS_GELU || EPI == EPI_DGELU)),
                  "wide tile: CTA pairs, one shard, store / bias+GeLU / GeLU' epilogues");
    constexpr int STAGES = C::STAGES;

    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[MAX_STAGES];
    __shared__ __align__(8) uint64_t bar_empty[MAX_STAGES];
    __shared__ __align__(8) uint64_t bar_tfull[2];
    __shared__ __align__(8) uint64_t bar_tempty[2];
    __shared__ __align__(8) uint64_t bar_done;
    __shared__ __align__(8) uint64_t bar_aux[EPI_THREADS / 32];
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_sh;

    const uint32_t smem_base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // In a pair the even CTA (rank 0) issues the MMAs and owns the barriers both
    // CTAs feed: the stage-full barriers (loads of both CTAs) and the
    // accumulator-empty barriers (epilogues of both CTAs).
    const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int unit_id = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int num_units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // one arrival (the leader's expect-tx for the stage bytes of the whole
            // pair) plus the transaction bytes of every copy into the stage
            ptx::mbar_init(ptx::smem_u32(&bar_full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&bar_empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_u32(&bar_tfull[b]), 1);
            // one arrival per epilogue warp of every CTA of the pair
            ptx::mbar_init(ptx::smem_u32(&bar_tempty[b]), (EPI_THREADS / 32) * CG);
        }
        ptx::mbar_init(ptx::smem_u32(&bar_done), 1);
        for (int w = 0; w < EPI_THREADS / 32; ++w) ptx::mbar_init(ptx::smem_u32(&bar_aux[w]), 1);
        abort_sh = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
        if constexpr (WIDE) ptx::prefetch_tensormap(&tmB2);
        ptx::prefetch_tensormap(&tmO0);
        ptx::prefetch_tensormap(&tmO1);
        ptx::prefetch_tensormap(&tmO2);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            ptx::tmem_alloc_pair(ptx::smem_u32(&tmem_base_sh), TMEM_COLS);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(ptx::smem_u32(&tmem_base_sh), TMEM_COLS);
            ptx::tmem_relinquish();
        }
    }
    ptx::tc_fence_before();
    if constexpr (PAIR)
        ptx::cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
    else
        __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = tmem_base_sh;
    // Programmatic dependent launch: the set-up above touched only on-chip state
    // and may overlap the previous kernel's tail; global memory is used only
    // after that kernel's grid has completed.
    ptx::griddep_wait();
    // Debug build: the dynamic shared memory of the launch holds the aligned ring
    // and the staging boxes, and the tile counts are positive.
    const uint32_t ring_end = smem_base + STAGES * C::STAGE_BYTES;
    const uint32_t stg_end = ring_end + (EPI_THREADS / 32) * C::STG_PER_WARP;
    const bool launch_ok = dbg_ok(stg_end <= ptx::smem_u32(smem_raw) + dynamic_smem_bytes() && p.m_tiles > 0 &&
                                      p.n_tiles > 0 && p.batch > 0 && p.nshards > 0 && p.kb_per_shard > 0,
                                  p, &abort_sh, 0x0100u);
    (void)ring_end, (void)stg_end;

    const int num_tiles = p.m_tiles * p.n_tiles * p.batch + (WIDE ? p.wide_tail : 0);

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = launch_ok;
            if constexpr (WIDE) {
            // Wide tiles: A as in the other tiles; B is this CTA's 256 of the tile's
            // 512 columns (one copy, map tmB), or for a half-width slot the 128 of
            // them in that half (map tmB2), placed where the MMA of that half reads.
            for (int tile = unit_id; tile < num_tiles && ok; tile += num_units) {
                int mb, nb, zb, hm;
                wide_coords(tile, p, mb, nb, zb, hm);
                const int m0 = mb * C::TILE_M + BM * static_cast<int>(rank);
                const int hs = hm == 2 ? 1 : 0;  // first half loaded
                const bool both = hm == 3;
                const int n0 = nb * TILE_N + C::B_ROWS * static_cast<int>(rank) + (C::B_ROWS / 2) * hs;
                const uint32_t stage_bytes = CG * (C::A_STAGE + (both ? C::B_STAGE : C::B_STAGE / 2));
                const int b_blocks = (both ? C::B_ROWS : C::B_ROWS / 2) / 64;
                const CUtensorMap *bmap = both ? &tmB : &tmB2;
                const bool ones_tile = EPI == EPI_STORE && A_MN && B_MN && p.bias_tile && mb == p.m_tiles - 1;
                const int nkb = p.kb_per_shard;
                const bool down = p.serpentine && ((tile / num_units) & 1);
                if (!dbg_ok(mb >= 0 && mb < p.m_tiles && nb >= 0 && nb < p.n_tiles && zb >= 0 && zb < p.batch &&
                                (hm == 1 || hm == 2 || hm == 3) && n0 % 64 == 0,
                            p, &abort_sh, 0x0201u)) {
                    ok = false;
                    break;
                }
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!ptx::mbar_wait_scoped<false>(ptx::smem_u32(&bar_empty[stage]), phase ^ 1u, p.wait_ns,
                                                     &abort_sh)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full_local = ptx::smem_u32(&bar_full[stage]);
                    const uint32_t full = ptx::mapa_shared(full_local, 0);
                    const uint32_t sa = smem_base + stage * C::STAGE_BYTES;
                    const uint32_t sb = sa + C::A_STAGE + hs * (C::B_STAGE / 2);
                    const int k0 = (down ? nkb - 1 - kb : kb) * BK;
                    if (!dbg_ok(stage >= 0 && stage < STAGES && sb + b_blocks * MN_BLOCK_BYTES <= ring_end &&
                                    k0 >= 0 && k0 < nkb * BK,
                                p, &abort_sh, 0x0301u)) {
                        ok = false;
                        break;
                    }
                    if (leader) ptx::mbar_arrive_expect_tx(full_local, stage_bytes);
                    if (ones_tile) {
                        // the bias-gradient tile: A is the 64 x 64 block of ones (rank 0,
                        // block 0), the rest reads as zero (see the other tiles' loop)
#pragma unroll
                        for (int j = 0; j < BM / 64; ++j)
                            ptx::tma_load_3d_pair(sa + j * MN_BLOCK_BYTES, &tmO2, full,
                                                  BM * static_cast<int>(rank) + 64 * j, 0, 0);
                    } else if constexpr (!A_MN) {
                        ptx::tma_load_3d_pair(sa, &tmA, full, k0, m0, zb);
                    } else {
                        if (p.a_mn4) {
                            ptx::tma_load_4d_pair(sa, &tmA, full, 0, k0, m0 / 64, zb);
                        } else {
#pragma unroll
                            for (int j = 0; j < BM / 64; ++j)
                                ptx::tma_load_3d_pair(sa + j * MN_BLOCK_BYTES, &tmA, full, m0 + 64 * j, k0, zb);
                        }
                    }
                    if constexpr (!B_MN) {
                        ptx::tma_load_3d_pair(sb, bmap, full, k0, n0, zb);
                    } else {
                        if (p.b_mn4) {
                            ptx::tma_load_4d_pair(sb, bmap, full, 0, k0, n0 / 64, zb);
                        } else {
                            for (int j = 0; j < b_blocks; ++j)
                                ptx::tma_load_3d_pair(sb + j * MN_BLOCK_BYTES, &tmB, full, n0 + 64 * j, k0, zb);
                        }
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            } else {
            for (int tile = unit_id; tile < num_tiles && ok; tile += num_units) {
                int mb, nb, zb;
                tile_coords(tile, p, mb, nb, zb);
                if (!tile_active<C::TILE_M, C::TILE_N>(p, mb, nb)) continue;
                const int m0 = mb * C::TILE_M + BM * static_cast<int>(rank);
                const int n0 = nb * TILE_N + C::B_ROWS * static_cast<int>(rank);
                int kb0, kb1;
                k_range<C::TILE_M>(p, mb, kb0, kb1);
                if (!dbg_ok(mb >= 0 && mb < p.m_tiles && nb >= 0 && nb < p.n_tiles && zb >= 0 && zb < p.batch &&
                                kb0 >= 0 && kb0 <= kb1 && kb1 <= p.nshards * p.kb_per_shard && n0 % 64 == 0,
                            p, &abort_sh, 0x0401u)) {
                    ok = false;
                    break;
                }
                if constexpr (EPI == EPI_STORE && A_MN && B_MN && !HEADS) {
                    if (p.bias_tile && mb == p.m_tiles - 1) {
                        // The ones tile (its own loop, so the main loop below is unchanged):
                        // A's columns 0..63 are ones (rank 0, block 0), the rest read as
                        // zero; the same 64 x 64 block serves every k-block, since rows
                        // past K meet zero-filled B rows.
                        for (int kb = kb0; kb < kb1 && ok; ++kb) {
                            if (!ptx::mbar_wait_scoped<false>(ptx::smem_u32(&bar_empty[stage]), phase ^ 1u,
                                                             p.wait_ns, &abort_sh)) {
                                ok = false;
                                break;
                            }
                            const uint32_t full_local = ptx::smem_u32(&bar_full[stage]);
                            const uint32_t full = PAIR ? ptx::mapa_shared(full_local, 0) : full_local;
                            const uint32_t sa = smem_base + stage * C::STAGE_BYTES;
                            const uint32_t sb = sa + C::A_STAGE;
                            if (leader) ptx::mbar_arrive_expect_tx(full_local, CG * C::STAGE_BYTES);
#pragma unroll
                            for (int j = 0; j < BM / 64; ++j) {
                                const int x = BM * static_cast<int>(rank) + 64 * j;
                                if constexpr (PAIR)
                                    ptx::tma_load_3d_pair(sa + j * MN_BLOCK_BYTES, &tmO2, full, x, 0, 0);
                                else
                                    ptx::tma_load_3d(sa + j * MN_BLOCK_BYTES, &tmO2, full, x, 0, 0);
                            }
                            // B exactly as in the main loop: one 4-D copy, or one per block
                            if (p.b_mn4) {
                                if constexpr (PAIR)
                                    ptx::tma_load_4d_pair(sb, &tmB, full, 0, kb * BK, n0 / 64, zb);
                                else
                                    ptx::tma_load_4d(sb, &tmB, full, 0, kb * BK, n0 / 64, zb);
                            } else {
#pragma unroll
                                for (int j = 0; j < C::B_ROWS / 64; ++j) {
                                    if constexpr (PAIR)
                                        ptx::tma_load_3d_pair(sb + j * MN_BLOCK_BYTES, &tmB, full, n0 + 64 * j,
                                                              kb * BK, zb);
                                    else
                                        ptx::tma_load_3d(sb + j * MN_BLOCK_BYTES, &tmB, full, n0 + 64 * j, kb * BK,
                                                         zb);
                                }
                            }
                            ++issued;
                            if (++stage == STAGES) {
                                stage = 0;
                                phase ^= 1u;
                            }
                        }
                        continue;
                    }
                }
                // Odd waves walk the tile's K range downwards (serpentine): for a
                // shard fold, the shards in descending order, each from its last
                // k-block; the MMA and the fold take the units in the order they come.
                const bool down = !HEADS && p.serpentine && ((tile / num_units) & 1);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!ptx::mbar_wait_scoped<false>(ptx::smem_u32(&bar_empty[stage]), phase ^ 1u, p.wait_ns,
                                                     &abort_sh)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full_local = ptx::smem_u32(&bar_full[stage]);
                    const uint32_t full = PAIR ? ptx::mapa_shared(full_local, 0) : full_local;
                    const uint32_t sa = smem_base + stage * C::STAGE_BYTES;
                    const uint32_t sb = sa + C::A_STAGE;
                    const int k0 = (down ? kb0 + kb1 - 1 - kb : kb) * BK;
                    if (!dbg_ok(stage >= 0 && stage < STAGES && sb + C::B_STAGE <= ring_end, p, &abort_sh, 0x0501u)) {
                        ok = false;
                        break;
                    }
                    auto load = [&](uint32_t dst, const CUtensorMap *map, int x, int y) {
                        if constexpr (PAIR)
                            ptx::tma_load_3d_pair(dst, map, full, x, y, zb);
                        else
                            ptx::tma_load_3d(dst, map, full, x, y, zb);
                    };
                    // one copy of every 64-wide MN block of the stage: (0, k, block, problem)
                    auto load4 = [&](uint32_t dst, const CUtensorMap *map, int k, int blk) {
                        if constexpr (PAIR)
                            ptx::tma_load_4d_pair(dst, map, full, 0, k, blk, zb);
                        else
                            ptx::tma_load_4d(dst, map, full, 0, k, blk, zb);
                    };
                    // The leader announces the bytes of both CTAs' copies; the peer's
                    // copies only complete bytes on the leader's barrier (they can land
                    // before the announcement: the phase still needs the arrival).
                    if (leader) ptx::mbar_arrive_expect_tx(full_local, CG * C::STAGE_BYTES);
                    if constexpr (HEADS) {
                        // per-head operands addressed in place (rank-3/4/5 maps)
                        int a2, a3, a4, b2, b3, b4;
                        head_coords(p.a_rank, zb, p.heads, p.hpt, a2, a3, a4);
                        head_coords(p.b_rank, zb, p.heads, p.hpt, b2, b3, b4);
                        if constexpr (!A_MN) {
                            tma_load_rank<PAIR>(sa, &tmA, full, k0, m0, p.a_rank, a2, a3, a4);
                        } else {
#pragma unroll
                            for (int j = 0; j < BM / 64; ++j)
                                tma_load_rank<PAIR>(sa + j * MN_BLOCK_BYTES, &tmA, full, m0 + 64 * j, k0, p.a_rank, a2,
                                                    a3, a4);
                        }
                        if constexpr (!B_MN) {
                            tma_load_rank<PAIR>(sb, &tmB, full, k0, n0, p.b_rank, b2, b3, b4);
                        } else {
#pragma unroll
                            for (int j = 0; j < C::B_ROWS / 64; ++j)
                                tma_load_rank<PAIR>(sb + j * MN_BLOCK_BYTES, &tmB, full, n0 + 64 * j, k0, p.b_rank,
                                                    b2, b3, b4);
                        }
                    } else {
                    if constexpr (!A_MN) {
                        load(sa, &tmA, k0, m0);
                    } else if (p.a_mn4) {
                        load4(sa, &tmA, k0, m0 / 64);
                    } else {
#pragma unroll
                        for (int j = 0; j < BM / 64; ++j) load(sa + j * MN_BLOCK_BYTES, &tmA, m0 + 64 * j, k0);
                    }
                    if constexpr (!B_MN) {
                        load(sb, &tmB, k0, n0);
                    } else if (p.b_mn4) {
                        load4(sb, &tmB, k0, n0 / 64);
                    } else {
#pragma unroll
                        for (int j = 0; j < C::B_ROWS / 64; ++j)
                            load(sb + j * MN_BLOCK_BYTES, &tmB, n0 + 64 * j, k0);
                    }
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            }
            if (!ok) record_timeout(p, &abort_sh, 1);
            // Let every copy started for this CTA's stages land before the CTA can
            // exit.  In a pair the stage-full barriers live in the leader and count
            // both CTAs' copies; the peer is held by the closing cluster barrier.
            if (leader) {
                const int64_t tail = issued < STAGES ? issued : STAGES;
                for (int64_t i = issued - tail; i < issued; ++i) {
                    const int s = static_cast<int>(i % STAGES);
                    const uint32_t ph = static_cast<uint32_t>((i / STAGES) & 1);
                    if (!ptx::mbar_wait_scoped<false>(ptx::smem_u32(&bar_full[s]), ph, p.wait_ns, nullptr))
                        record_timeout(p, &abort_sh, 2);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t unit = 0;
            bool ok = launch_ok;
            if constexpr (WIDE) {
            // Wide tiles: one accumulator of 512 columns, half h at TMEM columns
            // [256h, 256h + 256), filled by the MMAs of half h (B columns at
            // 16 KB * h in the stage).  A tile waits for the epilogue to drain each
            // half of the previous tile separately: it issues the first half's MMAs
            // for up to STAGES k-blocks (the stages already loaded) as soon as the
            // first half is drained, while the epilogue still drains the second
            // half, then the second half's MMAs of those k-blocks, then both halves
            // per k-block.  One commit per tile tells the epilogue the whole
            // accumulator is complete.
            uint32_t use[2] = {0u, 0u};
            auto issue_half = [&](int st, int hh, bool first) {
                const uint32_t sa = smem_base + st * C::STAGE_BYTES;
                const uint32_t sb = sa + C::A_STAGE + hh * (C::B_STAGE / 2);
                const uint32_t d_tmem = tmem_base + hh * MMA_N;
                if (!dbg_ok(st >= 0 && st < STAGES && (hh == 0 || hh == 1) && hh * MMA_N + MMA_N <= int(TMEM_COLS) &&
                                sb + C::B_STAGE / 2 <= ring_end,
                            p, &abort_sh, 0x0602u))
                    return;
#pragma unroll
                for (int k = 0; k < BK / 16; ++k) {
                    const uint64_t ad = A_MN ? ptx::sdesc_sw128(sa + k * 2048, MN_BLOCK_BYTES, 1024)
                                             : ptx::sdesc_sw128(sa + k * 32, 16, 1024);
                    const uint64_t bd = B_MN ? ptx::sdesc_sw128(sb + k * 2048, MN_BLOCK_BYTES, 1024)
                                             : ptx::sdesc_sw128(sb + k * 32, 16, 1024);
                    ptx::umma_f16_ss_pair(d_tmem, ad, bd, IDESC, (first && k == 0) ? 0u : 1u);
                }
            };
            auto wait_drained = [&](int hh) -> bool {
                const bool got = ptx::mbar_wait_scoped<false>(ptx::smem_u32(&bar_tempty[hh]), (use[hh] & 1u) ^ 1u,
                                                             p.wait_ns, &abort_sh);
                ++use[hh];
                ptx::tc_fence_after();
                return got;
            };
            auto wait_loaded = [&](int st, uint32_t ph) -> bool {
                const bool got = ptx::mbar_wait_scoped<false>(ptx::smem_u32(&bar_full[st]), ph, p.wait_ns, &abort_sh);
                ptx::tc_fence_after();
                return got;
            };
            auto release_stage = [&]() {
                ptx::umma_commit_pair_multicast(ptx::smem_u32(&bar_empty[stage]), 0x3);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            };
            for (int tile = unit_id; tile < num_tiles && ok; tile += num_units) {
                int mb, nb, zb, hm;
                wide_coords(tile, p, mb, nb, zb, hm);
                const int nkb = p.kb_per_shard;
                if (hm == 3) {
                    if (!wait_drained(0)) {
                        ok = false;
                        break;
                    }
                    const int lead = nkb < STAGES ? nkb : STAGES;
                    int st = stage;
                    uint32_t ph = phase;
                    for (int j = 0; j < lead; ++j) {
                        if (!wait_loaded(st, ph)) {
                            ok = false;
                            break;
                        }
                        issue_half(st, 0, j == 0);
                        if (++st == STAGES) st = 0, ph ^= 1u;
                    }
                    if (!ok || !wait_drained(1)) {
                        ok = false;
                        break;
                    }
                    for (int j = 0; j < lead; ++j) {
                        issue_half(stage, 1, j == 0);
                        release_stage();
                    }
                    for (int kb = lead; kb < nkb; ++kb) {
                        if (!wait_loaded(stage, phase)) {
                            ok = false;
                            break;
                        }
                        issue_half(stage, 0, false);
                        issue_half(stage, 1, false);
                        release_stage();
                    }
                } else {
                    const int hh = hm >> 1;  // the one half this slot computes
                    if (!wait_drained(hh)) {
                        ok = false;
                        break;
                    }
                    for (int kb = 0; kb < nkb; ++kb) {
                        if (!wait_loaded(stage, phase)) {
                            ok = false;
                            break;
                        }
                        issue_half(stage, hh, kb == 0);
                        release_stage();
                    }
                }
                if (!ok) break;
                ptx::umma_commit_pair_multicast(ptx::smem_u32(&bar_tfull[0]), 0x3);
            }
            } else {
            for (int tile = unit_id; tile < num_tiles && ok; tile += num_units) {
                int mb, nb, zb;
                tile_coords(tile, p, mb, nb, zb);
                if (!tile_active<C::TILE_M, C::TILE_N>(p, mb, nb)) continue;
                int kb0, kb1;
                k_range<C::TILE_M>(p, mb, kb0, kb1);
                // one shard: the tile's k-block range; several: kb_per_shard blocks each
                if (p.nshards > 1) kb0 = 0, kb1 = p.kb_per_shard;
                for (int s = 0; s < p.nshards && ok; ++s, ++unit) {
                    const uint32_t buf = unit & 1u, use = unit >> 1;
                    if (!ptx::mbar_wait_scoped<false>(ptx::smem_u32(&bar_tempty[buf]), (use & 1u) ^ 1u, p.wait_ns,
                                                     &abort_sh)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * TILE_N;
                    if (!dbg_ok(buf * TILE_N + TILE_N <= TMEM_COLS && kb0 >= 0 && kb0 <= kb1 &&
                                    kb1 <= p.nshards * p.kb_per_shard,
                                p, &abort_sh, 0x0702u)) {
                        ok = false;
                        break;
                    }
                    // Stages are taken two at a time: wait for both, then issue their
                    // eight MMAs back to back.  Measured on GB300 this issues 2-7% faster
                    // per clock than one stage at a time (MN/MN GEMMs gain once their
                    // operands come in one 4-D copy per stage).
                    for (int kb = kb0; kb < kb1;) {
                        const int nst = (kb + 1 < kb1) ? 2 : 1;
                        int st2 = stage + 1;
                        uint32_t ph2 = phase;
                        if (st2 == STAGES) st2 = 0, ph2 ^= 1u;
                        if (!ptx::mbar_wait_scoped<false>(ptx::smem_u32(&bar_full[stage]), phase, p.wait_ns,
                                                         &abort_sh)) {
                            ok = false;
                            break;
                        }
                        if (nst == 2 &&
                            !ptx::mbar_wait_scoped<false>(ptx::smem_u32(&bar_full[st2]), ph2, p.wait_ns, &abort_sh)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        for (int q = 0; q < nst; ++q) {
                            const int kk = kb + q;
                            const uint32_t sa = smem_base + stage * C::STAGE_BYTES;
                            const uint32_t sb = sa + C::A_STAGE;
#pragma unroll
                            for (int k = 0; k < BK / 16; ++k) {
                                const uint64_t ad = A_MN ? ptx::sdesc_sw128(sa + k * 2048, MN_BLOCK_BYTES, 1024)
                                                         : ptx::sdesc_sw128(sa + k * 32, 16, 1024);
                                const uint64_t bd = B_MN ? ptx::sdesc_sw128(sb + k * 2048, MN_BLOCK_BYTES, 1024)
                                                         : ptx::sdesc_sw128(sb + k * 32, 16, 1024);
                                const uint32_t acc = (kk != kb0 || k != 0) ? 1u : 0u;
                                if constexpr (PAIR)
                                    ptx::umma_f16_ss_pair(d_tmem, ad, bd, IDESC, acc);
                                else
                                    ptx::umma_f16_ss(d_tmem, ad, bd, IDESC, acc);
                            }
                            if constexpr (PAIR)
                                ptx::umma_commit_pair_multicast(ptx::smem_u32(&bar_empty[stage]), 0x3);
                            else
                                ptx::umma_commit(ptx::smem_u32(&bar_empty[stage]));
                            if (++stage == STAGES) {
                                stage = 0;
                                phase ^= 1u;
                            }
                        }
                        kb += nst;
                    }
                    if (!ok) break;
                    if constexpr (PAIR)
                        ptx::umma_commit_pair_multicast(ptx::smem_u32(&bar_tfull[buf]), 0x3);
                    else
                        ptx::umma_commit(ptx::smem_u32(&bar_tfull[buf]));
                }
            }
            }
            if (!ok) record_timeout(p, &abort_sh, 3);
            // Retire every MMA this thread issued before TMEM can be freed.
            if constexpr (PAIR)
                ptx::umma_commit_pair(ptx::smem_u32(&bar_done));
            else
                ptx::umma_commit(ptx::smem_u32(&bar_done));
            if (!ptx::mbar_wait(ptx::smem_u32(&bar_done), 0, p.wait_ns, nullptr)) record_timeout(p, &abort_sh, 4);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 2;                         // 0..7
        const int quarter = warp & 3;                    // TMEM lanes this warp may read
        const int half = ew >> 2;                        // column half of the tile
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t stg = smem_base + STAGES * C::STAGE_BYTES + ew * C::STG_PER_WARP;
        uint32_t unit = 0;
        bool ok = launch_ok;
        float sum[FOLD ? TILE_N / 2 : 1];
        (void)sum;
        AuxLoad aux{ptx::smem_u32(&bar_aux[ew]), 0u, false};
        // After every lane's tcgen05.ld of the buffer has completed, one arrival
        // per warp on the leader's accumulator-empty barrier.
        auto release = [&](uint32_t buf) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                const uint32_t a = ptx::smem_u32(&bar_tempty[buf]);
                if constexpr (PAIR)
                    ptx::mbar_arrive_remote(ptx::mapa_shared(a, 0));
                else
                    ptx::mbar_arrive(a);
            }
        };
        if constexpr (WIDE) {
        // Wide tiles: this warp finishes TMEM columns [128 * half, 128 * half + 128)
        // of each accumulator half hh; chunk q = 4 hh + c (c = 0..3) is output
        // columns 512 nb + 256 half + 32 q.  (The pair MMA of half hh reads B
        // columns 512 nb + 128 hh + [0, 128) in the even CTA and 512 nb + 256 +
        // 128 hh + [0, 128) in the odd one.)  Each half is released as soon as its
        // four chunks are in registers, so the next tile's MMAs of that half can
        // start.
        uint32_t tcount = 0;
        for (int tile = unit_id; tile < num_tiles && ok; tile += num_units) {
            if (tile + num_units >= num_tiles) ptx::griddep_launch_dependents();
            int mb, nb, zb, hm;
            wide_coords(tile, p, mb, nb, zb, hm);
            const int row0 = mb * C::TILE_M + BM * static_cast<int>(rank) + quarter * 32;
            const int64_t row = static_cast<int64_t>(row0) + lane;
            const int col0 = nb * TILE_N + half * (TILE_N / 2);
            const int qa = hm == 2 ? 4 : 0, qb = hm == 1 ? 4 : 8;
            const bool ones_tile = EPI == EPI_STORE && A_MN && B_MN && p.bias_tile && mb == p.m_tiles - 1;
            if constexpr (EPI == EPI_DGELU) aux_issue(&tmO1, aux, stg + STG_BOX, col0 + 32 * qa, row0, zb, lane);
            // The bias of each chunk is fetched one chunk ahead (the first while
            // the accumulator is still being computed).
            BiasPre bias_next;
            if constexpr (EPI == EPI_BIAS_GELU) bias_fetch(p.bias, col0 + 32 * qa, p.N, bias_next);
            bool got = ptx::mbar_wait_scoped<false>(ptx::smem_u32(&bar_tfull[0]), tcount & 1u, p.wait_ns, &abort_sh);
            ++tcount;
            got = __all_sync(0xffffffffu, got);
            if (!got) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            for (int q = qa; q < qb; ++q) {
                const uint32_t taddr = tmem_base + lane_off + (q >> 2) * MMA_N + half * 128 + (q & 3) * 32;
                if (!dbg_ok((q >> 2) * MMA_N + half * 128 + (q & 3) * 32 + 32 <= int(TMEM_COLS) &&
                                stg + C::STG_PER_WARP <= stg_end && (col0 + 32 * q) % 32 == 0 && row0 % 32 == 0,
                            p, &abort_sh, 0x0803u)) {
                    ok = false;
                    break;
                }
                BiasPre bias_cur;
                if constexpr (EPI == EPI_BIAS_GELU) {
                    bias_cur = bias_next;
                    if (q + 1 < qb) bias_fetch(p.bias, col0 + 32 * (q + 1), p.N, bias_next);
                }
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(taddr, r);
                ptx::tmem_ld_wait(r);
                if ((q & 3) == 3) release(static_cast<uint32_t>(q >> 2));
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                if (ones_tile) {
                    // row 0 of the ones tile holds the column sums of B; the tile
                    // has no rows of the output
                    if (rank == 0 && quarter == 0 && lane == 0) store_bias_grad(p, col0 + 32 * q, v);
                    continue;
                }
                finish_chunk<EPI, false>(p, &tmO0, &tmO1, &tmO2, v, row, row0, col0 + 32 * q, zb, lane, stg, &aux,
                                         q + 1 < qb ? col0 + 32 * (q + 1) : -1, row0, &abort_sh,
                                         EPI == EPI_BIAS_GELU ? &bias_cur : nullptr);
            }
        }
        } else {
        for (int tile = unit_id; tile < num_tiles && ok; tile += num_units) {
            // On starting this CTA's last tile, allow the next kernel in the stream
            // to be scheduled: its CTAs take the SMs of CTAs that have finished.
            // Only CTAs already running get here, so the next kernel can never
            // hold SMs that a CTA of this grid still waits for.
            if (tile + num_units >= num_tiles) ptx::griddep_launch_dependents();
            int mb, nb, zb;
            tile_coords(tile, p, mb, nb, zb);
            if (!tile_active<C::TILE_M, C::TILE_N>(p, mb, nb)) continue;
            const int row0 = mb * C::TILE_M + BM * static_cast<int>(rank) + quarter * 32;
            const int64_t row = static_cast<int64_t>(row0) + lane;
            const int col0 = nb * TILE_N + half * (TILE_N / 2);
            if constexpr (EPI == EPI_DGELU) aux_issue(&tmO1, aux, stg + STG_BOX, col0, row0, zb, lane);
            if constexpr (EPI == EPI_ATTN_DS) aux_issue(&tmO1, aux, stg + STG_BOX_WIDE, col0, row0, zb, lane, STG_BOX_WIDE);
            for (int s = 0; s < p.nshards; ++s, ++unit) {
                const uint32_t buf = unit & 1u, use = unit >> 1;
                bool got = ptx::mbar_wait_scoped<false>(ptx::smem_u32(&bar_tfull[buf]), use & 1u, p.wait_ns,
                                                       &abort_sh);
                got = __all_sync(0xffffffffu, got);
                if (!got) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t taddr = tmem_base + lane_off + buf * TILE_N + half * (TILE_N / 2);
                if (!dbg_ok(buf * TILE_N + TILE_N <= TMEM_COLS && stg + C::STG_PER_WARP <= stg_end &&
                                col0 % 32 == 0 && row0 % 32 == 0 && mb >= 0 && mb < p.m_tiles && nb >= 0 &&
                                nb < p.n_tiles && zb >= 0 && zb < p.batch,
                            p, &abort_sh, 0x0903u)) {
                    ok = false;
                    break;
                }
                if constexpr (FOLD) {
#pragma unroll
                    for (int c = 0; c < CHUNKS; ++c) {
                        uint32_t r[32];
                        ptx::tmem_ld_32x32b_x32(taddr + c * 32, r);
                        ptx::tmem_ld_wait(r);
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float v = __uint_as_float(r[i]);
                            sum[c * 32 + i] = (s == 0) ? v : sum[c * 32 + i] + v;
                        }
                    }
                    release(buf);
                    if (s == p.nshards - 1) {
#pragma unroll
                        for (int c = 0; c < CHUNKS; ++c) {
                            float v[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = sum[c * 32 + i];
                            finish_chunk<EPI, HEADS>(p, &tmO0, &tmO1, &tmO2, v, row, row0, col0 + c * 32, zb, lane, stg);
                        }
                    }
                } else {
                    if (EPI == EPI_STORE && A_MN && B_MN && p.bias_tile && mb == p.m_tiles - 1) {
                        // The ones tile: its row 0 holds the column sums of B; it has no
                        // rows of the output (all of them lie past M).
                        for (int c = 0; c < CHUNKS; ++c) {
                            uint32_t r[32];
                            ptx::tmem_ld_32x32b_x32(taddr + c * 32, r);
                            ptx::tmem_ld_wait(r);
                            if (c == CHUNKS - 1) release(buf);
                            if (rank == 0 && quarter == 0 && lane == 0) {
                                float v[32];
#pragma unroll
                                for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                                store_bias_grad(p, col0 + c * 32, v);
                            }
                        }
                        continue;
                    }
                    if constexpr (EPI == EPI_ATTN_DS) {
                        // Chunks in pairs: one P load and one dS store per 64 columns.
                        const uint32_t sbox = stg, pbox = stg + STG_BOX_WIDE;
#pragma unroll
                        for (int q = 0; q < CHUNKS / 2; ++q) {
                            const int colq = col0 + 64 * q;
                            const bool landed = ptx::mbar_wait(aux.bar, aux.phase, p.wait_ns, &abort_sh);
                            aux.phase ^= 1u;
                            aux.pending = false;
                            if (!__all_sync(0xffffffffu, landed) && lane == 0) record_timeout(p, &abort_sh, 6);
#pragma unroll
                            for (int hf = 0; hf < 2; ++hf) {
                                const int c = 2 * q + hf;
                                uint32_t r[32];
                                ptx::tmem_ld_32x32b_x32(taddr + c * 32, r);
                                ptx::tmem_ld_wait(r);
                                if (c == CHUNKS - 1) release(buf);
                                float v[32];
#pragma unroll
                                for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                                if (hf == 0) {
                                    // the previous pair's store has left the store box
                                    if (lane == 0) ptx::bulk_wait_read0();
                                    __syncwarp();
                                }
                                ds_half(p, v, row, zb, lane, sbox, pbox, hf);
                            }
                            ptx::fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0 && row0 < p.M && colq < p.N) {
                                ptx::tma_store_3d(&tmO0, sbox, colq, row0, zb);
                                ptx::bulk_commit();
                            }
                            // the P box is free: the next pair's P, once this store has left its box
                            if (q + 1 < CHUNKS / 2)
                                aux_issue(&tmO1, aux, pbox, colq + 64, row0, zb, lane, STG_BOX_WIDE);
                        }
                    } else {
#pragma unroll
                    for (int c = 0; c < CHUNKS; ++c) {
                        uint32_t r[32];
                        ptx::tmem_ld_32x32b_x32(taddr + c * 32, r);
                        ptx::tmem_ld_wait(r);
                        // the whole accumulator slice is in registers: release the buffer
                        if (c == CHUNKS - 1) release(buf);
                        float v[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                        finish_chunk<EPI, HEADS>(p, &tmO0, &tmO1, &tmO2, v, row, row0, col0 + c * 32, zb, lane, stg, &aux,
                                          c < CHUNKS - 1 ? col0 + (c + 1) * 32 : -1, row0, &abort_sh);
                    }
                    }
                }
            }
        }
        }
        if (!ok) record_timeout(p, &abort_sh, 5);
        // an H or P load still in flight (only after an abort) must land before the CTA exits
        if (aux.pending && !ptx::mbar_wait(aux.bar, aux.phase, p.wait_ns, nullptr) && lane == 0)
            record_timeout(p, &abort_sh, 7);
        // every TMA store of this warp must be complete before the CTA exits
        if (lane == 0) ptx::bulk_wait0();
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    // In a pair, neither CTA leaves (or frees TMEM) while the leader's MMAs may
    // still read the peer's shared memory or write its TMEM.
    if constexpr (PAIR) ptx::cluster_sync();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        if constexpr (PAIR)
            ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else
            ptx::tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                                         cudaEnableDefault, &q);
        if (e == cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        else
            set_last_error("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled): %s, query %d",
                           cudaGetErrorString(e), static_cast<int>(q));
    });
    return fn;
}

// Row-major bf16 matrix [rows, cols] with a box of box_cols (inner) x box_rows.
// A batch of `batch` contiguous row-major [rows, cols] matrices is a 3-D tensor
// (cols, rows, batch); a plain matrix has batch 1.
static bool make_map(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols, uint32_t box_cols,
                     uint32_t box_rows, CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B, int64_t batch = 1,
                     CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    auto fn = encode_fn();
    if (!fn) {
        set_last_error("cuTensorMapEncodeTiled is not available from the driver");
        return false;
    }
    const cuuint64_t esz = dt == CU_TENSOR_MAP_DATA_TYPE_FLOAT32 ? 4 : 2;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * esz,
                             static_cast<cuuint64_t>(cols) * static_cast<cuuint64_t>(rows) * esz};
    cuuint32_t box[3] = {box_cols, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, dt, 3,
                    const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        set_last_error("cuTensorMapEncodeTiled failed (CUresult %d) for %lld x [%lld, %lld] matrices, box %u x %u",
                       static_cast<int>(r), static_cast<long long>(batch), static_cast<long long>(rows),
                       static_cast<long long>(cols), box_cols, box_rows);
    return r == CUDA_SUCCESS;
}

// An MN-major operand [K, MN] (MN contiguous, MN a multiple of 64) as the 4-D
// tensor (64, K, MN/64, batch): one copy brings `nblk` consecutive 64-wide MN
// blocks of `box_k` rows, laid out block after block in shared memory exactly
// as the per-block copies do.  The third dimension steps 128 bytes, inside the
// row pitch of the second; returns false if the driver does not take the map
// (the caller then keeps the per-block 3-D map).
static bool make_map_mn4(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols, uint32_t box_k,
                         uint32_t nblk, int64_t batch) {
    auto fn = encode_fn();
    if (!fn || cols % 64 != 0) return false;
    cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64),
                          static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(cols) * 2, 128,
                             static_cast<cuuint64_t>(cols) * static_cast<cuuint64_t>(rows) * 2};
    cuuint32_t box[4] = {64, box_k, nblk, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// A rank-4 or rank-5 view (see HeadView) with a box of box0 elements along d and
// box1 along S (1 in the head and batch dimensions).
static bool make_map_view(CUtensorMap *m, const void *ptr, const HeadView &v, uint32_t box0, uint32_t box1,
                          CUtensorMapSwizzle swz) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t e = 2;
    cuuint64_t dims[5], strides[4];
    cuuint32_t box[5] = {box0, box1, 1, 1, 1}, estr[5] = {1, 1, 1, 1, 1};
    int rank = 0;
    if (v.rank == 4) {
        rank = 4;
        const cuuint64_t d4[4] = {static_cast<cuuint64_t>(v.d), static_cast<cuuint64_t>(v.S),
                                  static_cast<cuuint64_t>(v.heads), static_cast<cuuint64_t>(v.nb)};
        const cuuint64_t s4[3] = {static_cast<cuuint64_t>(v.ld) * e, static_cast<cuuint64_t>(v.d) * e,
                                  static_cast<cuuint64_t>(v.S) * static_cast<cuuint64_t>(v.ld) * e};
        for (int i = 0; i < 4; ++i) dims[i] = d4[i];
        for (int i = 0; i < 3; ++i) strides[i] = s4[i];
    } else if (v.rank == 5) {
        rank = 5;
        const cuuint64_t d5[5] = {static_cast<cuuint64_t>(v.d), static_cast<cuuint64_t>(v.S),
                                  static_cast<cuuint64_t>(v.hpt), static_cast<cuuint64_t>(v.heads / v.hpt),
                                  static_cast<cuuint64_t>(v.nb)};
        const cuuint64_t s5[4] = {static_cast<cuuint64_t>(v.ld) * e, static_cast<cuuint64_t>(v.d) * e,
                                  static_cast<cuuint64_t>(v.coli) * e,
                                  static_cast<cuuint64_t>(v.S) * static_cast<cuuint64_t>(v.ld) * e};
        for (int i = 0; i < 5; ++i) dims[i] = d5[i];
        for (int i = 0; i < 4; ++i) strides[i] = s5[i];
    } else {
        return false;
    }
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        set_last_error("cuTensorMapEncodeTiled failed (CUresult %d) for a rank-%d head view", static_cast<int>(r),
                       rank);
    return r == CUDA_SUCCESS;
}

template <int EPI, bool A_MN, bool B_MN, int CG, bool HEADS = false, int TILE_N = BN>
static cudaError_t launch_t(const GemmArgs &g, int num_sms, cudaStream_t st) {
    using C = Cfg<CG, TILE_N, EPI>;
    auto kern = gemm_kernel<EPI, A_MN, B_MN, CG, HEADS, TILE_N>;
    // Per-device, once: the shared-memory opt-in, and for CTA pairs the number of
    // 2-CTA clusters that can be resident at once (the persistent grid size).
    static std::mutex mu;
    static bool attr_set[64] = {};
    static int max_clusters[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    // attr[0]: the CTA-pair cluster; attr[1]: programmatic dependent launch (the
    // kernel's set-up overlaps the previous kernel's tail; TPMLP_PDL=0 turns it
    // off, a tuning knob read per call).
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_DYN;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = CG > 1 ? 1 : 0;  // single CTAs launch without a cluster
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!attr_set[dev]) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_DYN);
            if (e != cudaSuccess) {
                set_last_error("cudaFuncSetAttribute(%d bytes of shared memory): %s", C::SMEM_DYN,
                               cudaGetErrorString(e));
                return e;
            }
            if (CG > 1) {
                cfg.gridDim = dim3(static_cast<unsigned>(num_sms / CG * CG), 1, 1);
                int n = 0;
                e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
                if (e != cudaSuccess || n < 1) {
                    set_last_error("cudaOccupancyMaxActiveClusters: %s (%d)", cudaGetErrorString(e), n);
                    return e != cudaSuccess ? e : cudaErrorLaunchOutOfResources;
                }
                max_clusters[dev] = n;
            } else {
                max_clusters[dev] = num_sms;
            }
            attr_set[dev] = true;
        }
    }

    CUtensorMap ma, mb;
    // A operand: K-major [M,K] with a 64 x 128 box, or MN-major [K,M] with 64 x 64 boxes.
    // B operand: this CTA's B_ROWS columns, K-major in one box or MN-major in 64-wide boxes.
    const int64_t nb = g.batch < 1 ? 1 : g.batch;
    const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
    // MN-major operands whose MN extent is a multiple of 64 take the 4-D map
    // (one copy per stage instead of one per 64-wide block); TPMLP_MN4=0 keeps
    // the per-block maps (a tuning knob, read per call).
    const char *mn4_env = std::getenv("TPMLP_MN4");
    const bool mn4 = !(mn4_env && mn4_env[0] == '0');
    // Per-head views (HEADS): K-major boxes of 64 (d) x rows, MN-major boxes of
    // 64 (d) x BK; the 4-D per-stage copy is not used for them.
    const int a_rank = HEADS && g.a_view.rank > 3 ? g.a_view.rank : 3;
    const int b_rank = HEADS && g.b_view.rank > 3 ? g.b_view.rank : 3;
    const int o_rank = HEADS && g.o_view.rank > 3 ? g.o_view.rank : 3;
    // (HEADS kernels always copy MN-major operands block by block.)
    constexpr bool WIDE = TILE_N == 512;
    CUtensorMap mb2;  // wide tiles: B of one 256-column half of the tile (half the box)
    const bool a4 = !HEADS && A_MN && mn4 && g.M % 64 == 0 && make_map_mn4(&ma, g.a, g.K, g.M, BK, BM / 64, nb);
    const bool b4 = !HEADS && B_MN && mn4 && g.N % 64 == 0 &&
                    make_map_mn4(&mb, g.b, g.K, g.N, BK, C::B_ROWS / 64, nb) &&
                    (!WIDE || make_map_mn4(&mb2, g.b, g.K, g.N, BK, C::B_ROWS / 128, nb));
    bool oka, okb;
    if (a_rank > 3)
        oka = make_map_view(&ma, g.a, g.a_view, 64, A_MN ? BK : BM, sw);
    else
        oka = a4 || (A_MN ? make_map(&ma, g.a, g.K, g.M, 64, BK, sw, nb) : make_map(&ma, g.a, g.M, g.K, BK, BM, sw, nb));
    if (b_rank > 3)
        okb = make_map_view(&mb, g.b, g.b_view, 64, B_MN ? BK : C::B_ROWS, sw);
    else
        okb = b4 || (B_MN ? make_map(&mb, g.b, g.K, g.N, 64, BK, sw, nb)
                          : make_map(&mb, g.b, g.N, g.K, BK, C::B_ROWS, sw, nb));
    if (WIDE && !B_MN && okb) okb = make_map(&mb2, g.b, g.N, g.K, BK, C::B_ROWS / 2, sw, nb);
    if (!WIDE || (B_MN && !b4)) mb2 = mb;  // unused, or the per-block maps serve both widths
    if (!oka || !okb) return cudaErrorInvalidValue;
    // Output maps: [M, N] row-major, 32 x 32 boxes, 64-byte swizzle (matches stage_row).
    // Bias + GeLU writes H (optional) and Y; GeLU' reads H through the second map;
    // the others write out0 only.
    // The GeLU' epilogue can also write Y rebuilt from H (third map).
    CUtensorMap mo0, mo1, mo2;
    const void *o0 = g.out0 ? g.out0 : g.out1;
    // The attention scores are fp16 (32 x 32 box, 64-byte swizzle, as the bf16
    // outputs); dS reads P through the second map; both of its maps have 32 x 64
    // boxes with 128-byte swizzle (see stage_half_row128).
    const void *o1 = (EPI == EPI_BIAS_GELU) ? (g.out1 ? g.out1 : o0)
                                            : ((EPI == EPI_DGELU || EPI == EPI_ATTN_DS) ? g.aux : o0);
    const void *o2 = (EPI == EPI_DGELU && g.out1) ? g.out1 : o0;
    const CUtensorMapDataType odt =
        EPI == EPI_ATTN_SCORE ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const bool wide = EPI == EPI_ATTN_DS;
    const uint32_t obox = wide ? 64 : 32;
    const CUtensorMapSwizzle so = wide ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (wide && (o_rank > 3 || g.nshards != 1)) {
        set_last_error("dS epilogue: a plain [problems][M][N] output and one shard only");
        return cudaErrorInvalidValue;
    }
    // The bias-gradient tile takes its A from a 64 x 64 block of ones (third map).
    const bool bias_tile = EPI == EPI_STORE && A_MN && B_MN && g.bias_grad != nullptr;
    if (bias_tile && (g.ones == nullptr || nb != 1 || g.nshards != 1 || g.causal_k != 0 || g.skip_upper)) {
        set_last_error("bias-gradient tile: needs the ones block, one problem, one shard, no causal ranges");
        return cudaErrorInvalidValue;
    }
    if (!(o_rank > 3 ? make_map_view(&mo0, o0, g.o_view, 32, 32, so)
                     : make_map(&mo0, o0, g.M, g.N, obox, 32, so, nb, odt)) ||
        !make_map(&mo1, o1, g.M, g.N, obox, 32, so, nb, odt) ||
        !(bias_tile ? make_map(&mo2, g.ones, 64, 64, 64, BK, CU_TENSOR_MAP_SWIZZLE_128B, 1)
                    : make_map(&mo2, o2, g.M, g.N, 32, 32, so, nb, odt)))
        return cudaErrorInvalidValue;

    Params p;
    p.M = static_cast<int>(g.M);
    p.N = static_cast<int>(g.N);
    p.m_tiles = static_cast<int>((g.M + C::TILE_M - 1) / C::TILE_M);
    p.n_tiles = static_cast<int>((g.N + TILE_N - 1) / TILE_N);
    p.raster_n = g.raster_n ? 1 : 0;
    {
        const int fast_tiles = p.raster_n ? p.n_tiles : p.m_tiles;
        p.group = g.group < 1 ? 1 : (g.group > fast_tiles ? fast_tiles : g.group);
    }
    p.nshards = g.nshards;
    p.kb_per_shard = static_cast<int>((g.kshard + BK - 1) / BK);
    p.out0 = g.out0;
    p.out1 = g.out1;
    p.aux = g.aux;
    p.bias = g.bias;
    p.status = g.status;
    p.wait_ns = g.wait_ns;
    p.colsum_part = g.colsum_part;
    p.batch = static_cast<int>(nb);
    p.scale = g.scale;
    p.causal = g.causal ? 1 : 0;
    p.rowvec = g.rowvec;
    p.causal_k = g.causal_k;
    p.a_mn4 = a4 ? 1 : 0;
    p.b_mn4 = b4 ? 1 : 0;
    p.a_rank = a_rank;
    p.b_rank = b_rank;
    p.o_rank = o_rank;
    {
        const HeadView &hv = g.a_view.rank > 3 ? g.a_view : (g.b_view.rank > 3 ? g.b_view : g.o_view);
        p.heads = hv.heads > 0 ? static_cast<int>(hv.heads) : 1;
        p.hpt = hv.hpt > 0 ? static_cast<int>(hv.hpt) : 1;
    }
    p.bias_tile = bias_tile ? 1 : 0;
    p.bias_grad = g.bias_grad;
    if (bias_tile) p.m_tiles += 1;  // the ones tile, after every row of the output
    p.skip_upper = g.skip_upper ? 1 : 0;
    // TPMLP_FLIP_ODD=0 keeps every problem's M-tiles in order (a tuning knob, read per call).
    {
        const char *flip = std::getenv("TPMLP_FLIP_ODD");
        p.flip_odd = (g.causal_k != 0 || g.skip_upper) && !(flip && flip[0] == '0') ? 1 : 0;
    }
    // TPMLP_PAIR_ORDER=0 keeps the reversed odd problems for the causal products
    // with one N-tile (a tuning knob, read per call).
    {
        const char *po = std::getenv("TPMLP_PAIR_ORDER");
        p.pair_order = g.causal_k != 0 && p.n_tiles == 1 && p.m_tiles % 2 == 0 && !(po && po[0] == '0') ? 1 : 0;
    }
    // The causal ranges are defined for square per-head problems in one shard.
    if ((g.causal_k != 0 || g.skip_upper) && (g.nshards != 1 || (g.causal_k != 0 && g.M != g.K))) {
        set_last_error("causal K ranges need one shard and M = K (M=%lld K=%lld, %d shards)",
                       static_cast<long long>(g.M), static_cast<long long>(g.K), g.nshards);
        return cudaErrorInvalidValue;
    }
    int tiles = p.m_tiles * p.n_tiles * p.batch;
    int resident = max_clusters[dev];
    if (const char *o = std::getenv("TPMLP_MAX_UNITS")) resident = std::atoi(o) > 0 ? std::atoi(o) : resident;
    // Wide tiles: a last partial wave of r tiles is run as 2r half-width tiles
    // when they fit in one wave (2r <= units): the wave then takes about half a
    // wide tile's time.  TPMLP_WIDE_TAIL=0 keeps whole tiles (a tuning knob, read
    // per call).
    p.wide_tail = 0;
    // TPMLP_SERPENTINE=0 walks K upwards in every wave (a tuning knob, read per call).
    {
        const char *se = std::getenv("TPMLP_SERPENTINE");
        p.serpentine = (WIDE || (!HEADS && g.causal_k == 0 && !g.skip_upper)) && !(se && se[0] == '0') ? 1 : 0;
    }
    if (WIDE) {
        const char *tail_env = std::getenv("TPMLP_WIDE_TAIL");
        const int r = tiles % resident;
        if (!(tail_env && tail_env[0] == '0') && 2 * r <= resident) p.wide_tail = r;
        tiles += p.wide_tail;
    }
    const int units = tiles < resident ? tiles : resident;
    p.units = units;
    if (std::getenv("TPMLP_DEBUG_LAUNCH"))
        std::fprintf(stderr, "tpmlp gemm epi=%d cg=%d M=%lld N=%lld K=%lld tiles=%d resident=%d grid=%d group=%d%c\n",
                     EPI, CG, static_cast<long long>(g.M), static_cast<long long>(g.N), static_cast<long long>(g.K),
                     tiles, max_clusters[dev], units * CG, p.group, p.raster_n ? 'n' : 'm');
    cfg.gridDim = dim3(static_cast<unsigned>(units * CG), 1, 1);
    const char *pdl_env = std::getenv("TPMLP_PDL");
    if (!(pdl_env && pdl_env[0] == '0')) {
        if (CG > 1) {
            cfg.attrs = attr;
            cfg.numAttrs = 2;
        } else {
            cfg.attrs = attr + 1;
            cfg.numAttrs = 1;
        }
    }
    e = cudaLaunchKernelEx(&cfg, kern, ma, mb, mo0, mo1, mo2, mb2, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        cudaFuncAttributes fa;
        std::memset(&fa, 0, sizeof(fa));
        cudaFuncGetAttributes(&fa, kern);
        set_last_error("tensor-core GEMM launch (grid %d x cluster %d, %d threads, %d bytes shared): %s "
                       "[kernel: %d regs, max %d threads, %zu static + max %d dynamic shared bytes]",
                       units, CG, NUM_THREADS, C::SMEM_DYN, cudaGetErrorString(e), fa.numRegs,
                       fa.maxThreadsPerBlock, fa.sharedSizeBytes, fa.maxDynamicSharedSizeBytes);
    }
    return e;
}

template <int EPI, bool A_MN, bool B_MN>
static cudaError_t launch_cg(const GemmArgs &g, int num_sms, cudaStream_t st) {
    if constexpr (EPI == EPI_BIAS_GELU || EPI == EPI_DGELU || (EPI == EPI_STORE && A_MN == B_MN)) {
        if (tc_wide_tile(static_cast<Epi>(EPI), g)) return launch_t<EPI, A_MN, B_MN, 2, false, 512>(g, num_sms, st);
    }
    if constexpr (EPI == EPI_STORE && !A_MN && !B_MN) {
        // plain products of two K-major operands (the attention's dO = dZ Wo^T)
        return g.cta_pair ? launch_t<EPI, false, false, 2>(g, num_sms, st) : launch_t<EPI, false, false, 1>(g, num_sms, st);
    } else {
    if constexpr (EPI == EPI_ATTN_SCORE || EPI == EPI_ATTN_DS || EPI == EPI_STORE) {
        if (g.heads_layout) {
            // Outputs at most 128 wide (the per-head products with N = d) take the
            // narrow tile: the wide one would spend half its MMA work on columns
            // past N.  TPMLP_NARROW=0 keeps the wide tile (a tuning knob, read per call).
            if constexpr (EPI == EPI_STORE) {
                const char *nar = std::getenv("TPMLP_NARROW");
                if (g.cta_pair && g.N <= 128 && !(nar && nar[0] == '0'))
                    return launch_t<EPI, A_MN, B_MN, 2, true, 128>(g, num_sms, st);
            }
            return g.cta_pair ? launch_t<EPI, A_MN, B_MN, 2, true>(g, num_sms, st)
                              : launch_t<EPI, A_MN, B_MN, 1, true>(g, num_sms, st);
        }
    }
    return g.cta_pair ? launch_t<EPI, A_MN, B_MN, 2>(g, num_sms, st) : launch_t<EPI, A_MN, B_MN, 1>(g, num_sms, st);
    }
}

}  // namespace tc

bool tc_wide_tile(Epi epi, const GemmArgs &g) {
    if (!g.cta_pair || g.heads_layout || g.nshards != 1 || g.causal_k != 0 || g.skip_upper) return false;
    if (!(epi == EPI_BIAS_GELU || epi == EPI_DGELU || (epi == EPI_STORE && g.a_mn == g.b_mn))) return false;
    const char *w = std::getenv("TPMLP_WIDE");
    return !(w && w[0] == '0');
}

cudaError_t launch_tc_gemm(Epi epi, const GemmArgs &g, int num_sms, cudaStream_t st) {
    using namespace tc;
    if (g.M <= 0 || g.N <= 0 || g.K <= 0) return cudaSuccess;
    switch (epi) {
        case EPI_BIAS_GELU:  // X[T,h] (K-major) . A[h,F] (MN-major)
            if (!g.a_mn && g.b_mn) return launch_cg<EPI_BIAS_GELU, false, true>(g, num_sms, st);
            break;
        case EPI_FOLD_BIAS:  // Y[T,F] (K-major) . B[F,h] (MN-major)
            if (!g.a_mn && g.b_mn) return launch_cg<EPI_FOLD_BIAS, false, true>(g, num_sms, st);
            break;
        case EPI_DGELU:  // dZ[T,h] (K-major) . B[F,h]^T (K-major)
            if (!g.a_mn && !g.b_mn) return launch_cg<EPI_DGELU, false, false>(g, num_sms, st);
            break;
        case EPI_STORE:  // Y^T . dZ and X^T . dY: both operands MN-major; P . V: K-major . MN-major;
                         // dZ . Wo^T: both K-major
            if (g.a_mn && g.b_mn) return launch_cg<EPI_STORE, true, true>(g, num_sms, st);
            if (!g.a_mn && g.b_mn) return launch_cg<EPI_STORE, false, true>(g, num_sms, st);
            if (!g.a_mn && !g.b_mn) return launch_cg<EPI_STORE, false, false>(g, num_sms, st);
            break;
        case EPI_ATTN_SCORE:  // Q[S,d] (K-major) . K[S,d]^T (K-major), per head
            if (!g.a_mn && !g.b_mn) return launch_cg<EPI_ATTN_SCORE, false, false>(g, num_sms, st);
            break;
        case EPI_ATTN_DS:  // dO[S,d] (K-major) . V[S,d]^T (K-major), per head
            if (!g.a_mn && !g.b_mn) return launch_cg<EPI_ATTN_DS, false, false>(g, num_sms, st);
            break;
        case EPI_FOLD:  // dY[T,F] (K-major) . A[h,F]^T (K-major)
            if (!g.a_mn && !g.b_mn) return launch_cg<EPI_FOLD, false, false>(g, num_sms, st);
            break;
    }
    return cudaErrorNotSupported;
}

}  // namespace tpmlp
