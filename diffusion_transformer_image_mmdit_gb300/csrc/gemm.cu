// Persistent tcgen05 GEMM for the block linears: Y = X W^T with fused epilogues.
//
// The linears of both block types (QKV, output projection, MLP in/out, the
// single block's fused D -> 3D + D_mlp and its 5D -> D output) are dense
// bf16 contractions with fp32 accumulation (Luminal blog, section "The AMD
// MI300X pipeline": all bf16 GEMMs accumulate in fp32, with bias epilogues).
//
// Structure (one CTA per SM, 320 threads, clusters of two CTAs = one CTA
// pair):
//   The pair computes the vertically adjacent 128x256 output tiles (m, n)
//   and (m + 1, n) with one stream of tcgen05.mma.cta_group::2 (M = 256,
//   N = 256): each CTA loads its own 128 rows of A and one 128-row half of
//   the 256-row W tile into its own shared memory (plain TMA tile loads),
//   and the MMA reads both CTAs' halves, so W crosses L2 -> SM once per pair
//   and the pair issues half the MMAs two independent CTAs would.
//   warp 0      TMA producer (both CTAs): its A tile 128x128 and its W half
//               128x128 per K block (two 128-byte-swizzled K slices each)
//               into a 3-stage ring (64 KB per stage; a K that ends in one
//               slice ends in a one-slice stage).  Both CTAs' loads complete on CTA 0's
//               full barrier (two arrivals with their byte counts).  CTA 0's
//               MMAs release a stage with one commit multicast to both CTAs'
//               empty barriers.
//   warp 1      allocates 512 TMEM columns (two 128x256 fp32 accumulators)
//               in both CTAs (one collective pair allocation); in CTA 0 it
//               issues the pair MMAs (M=256, N=256, K=16) from one elected
//               lane; the accumulator-ready commit goes to both CTAs.
//   warps 2-9   epilogue (both CTAs): tcgen05.ld of the finished
//               accumulator of this CTA's 128 rows (one TMEM lane = one
//               output row per thread; two warps per lane quadrant, one per
//               128-column half), fused bias / per-channel scale / GELU-tanh
//               / SwiGLU / gated fp32 residual / q-k RMSNorm + RoPE /
//               transposed V store, overlapping the next tile's MMAs; the
//               drained accumulator is handed back on CTA 0's barrier.  The
//               gated residual x += gate * value is a TMA reduce-add of the
//               staged products into x (the addition happens in L2), so the
//               epilogue never reads the residual.
#include <mutex>

#include "common.cuh"

namespace mmdit {

namespace {

constexpr int kEpiWarps = 8;  // two per TMEM lane quadrant, one per 128-column half
constexpr int kGemmThreads = 32 * (2 + kEpiWarps);
// A stage holds two K slices of one 128-byte swizzle row each (128 bf16 or
// 256 e4m3 K elements): per stage one full-barrier wait, eight pair MMAs
// and one release, where one-slice stages made the barrier round trips
// (wait, commit, the release forwarded to CTA 1) cost up to 8 % of the
// K = 3072 launches.  The last stage of a K not a multiple of two slices
// holds one.
constexpr int kRing = 3;                           // stages of the TMA ring (192 KB)
constexpr uint32_t kHalfA = kBM * kBK * 2;         // 16 KB: one K slice of this CTA's 128 rows of A
constexpr uint32_t kHalfB = (kBN / 2) * kBK * 2;   // 16 KB: one K slice of this CTA's half of the W tile
constexpr uint32_t kStageA = 2 * kHalfA;
constexpr uint32_t kStageB = 2 * kHalfB;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kEpiStageBytes = 4096;  // staging area of one epilogue warp
constexpr size_t kGemmSmem = 1024 + kRing * (kStageA + kStageB) + kEpiWarps * kEpiStageBytes + 256;
static_assert(kGemmSmem <= 232448, "GEMM shared memory above the 227 KB a CTA can have");

struct TileCoord {
  int seg, tm, tn;
  bool valid;  // false for the second tile of a pair past the last M tile
};

// Work unit t of a problem is a pair of M tiles (2 pm, 2 pm + 1) over all
// segments, at one N tile; CTA `rank` of the cluster takes M tile 2 pm + rank.
// Grouped raster: runs of group_m pairs sweep all N tiles with M fastest, so
// the clusters of one wave share A and W tiles in L2.  A missing second tile
// (odd M tile count) repeats the last real tile with its stores switched off,
// so both CTAs run the same K loop.
__device__ __forceinline__ TileCoord tile_coord(const GemmParams& p, int t, int rank) {
  const int total_m = p.n_seg * p.tiles_m;
  const int pairs_m = (total_m + 1) >> 1;
  const int per_group = p.group_m * p.tiles_n;
  const int g = t / per_group;
  const int first = g * p.group_m;
  const int gm = min(p.group_m, pairs_m - first);
  const int r = t - g * per_group;
  int mi = 2 * (first + r % gm) + rank;
  TileCoord c;
  c.valid = mi < total_m;
  if (!c.valid) mi = total_m - 1;
  c.seg = mi / p.tiles_m;
  c.tm = mi - c.seg * p.tiles_m;
  c.tn = r / gm;
  return c;
}

__device__ __forceinline__ void load_vec32(const float* __restrict__ src, float* v) {
  const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float4 t = __ldg(s4 + i);
    v[4 * i] = t.x, v[4 * i + 1] = t.y, v[4 * i + 2] = t.z, v[4 * i + 3] = t.w;
  }
}

// Reads 32 accumulator columns of this thread's row and applies the fp8
// row scale rs, the int8 / fp8 channel scale and the bias.
__device__ __forceinline__ void acc_chunk(uint32_t taddr, const GemmParams& p, int n, float* v, float rs = 1.0f) {
  uint32_t raw[32];
  MMDIT_TMEM_LD32(taddr, raw);
  tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(raw[i]) * rs;
  if (p.wscale) {
    float s[32];
    load_vec32(p.wscale + n, s);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] *= s[i];
  }
  if (p.bias) {
    float b[32];
    load_vec32(p.bias + n, b);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] += b[i];
  }
}

// ------------------------------------------------------------ epilogue I/O
// Each epilogue thread owns one output row (its TMEM lane) and produces 32
// consecutive columns at a time.  Stored directly, one warp instruction
// would touch 32 rows with 16 bytes each (half sectors).  Instead the warp
// passes the 32 x 32 chunk through its own 4 KB staging area in shared
// memory (16-byte slots XOR-swizzled by row, so both the row-wise writes and
// the column-wise reads are free of bank conflicts) and every global
// instruction covers whole 32-byte sectors: 8 rows x 64 bytes for bf16, 4
// rows x 128 bytes for fp32.  `row0` points at column n of the warp's first
// row; rows at or beyond `nrows` are not touched.
__device__ __forceinline__ void warp_store_bf16x32(uint8_t* stg, int lane, const float* v, uint16_t* row0,
                                                   long long ld, int nrows) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * c + 0], v[8 * c + 1]);
    w.y = pack_bf16x2(v[8 * c + 2], v[8 * c + 3]);
    w.z = pack_bf16x2(v[8 * c + 4], v[8 * c + 5]);
    w.w = pack_bf16x2(v[8 * c + 6], v[8 * c + 7]);
    *reinterpret_cast<uint4*>(stg + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) = w;
  }
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int rr = i * 8 + (lane >> 2), c = lane & 3;
    const uint4 w = *reinterpret_cast<const uint4*>(stg + rr * 64 + ((c ^ ((rr >> 1) & 3)) << 4));
    if (rr < nrows) *reinterpret_cast<uint4*>(row0 + rr * ld + c * 8) = w;
  }
  __syncwarp();
}

__device__ __forceinline__ void warp_store_f32x32(uint8_t* stg, int lane, const float* v, float* row0, long long ld,
                                                  int nrows) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<float4*>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) =
        make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int rr = i * 4 + (lane >> 3), c = lane & 7;
    const float4 w = *reinterpret_cast<const float4*>(stg + rr * 128 + ((c ^ (rr & 7)) << 4));
    if (rr < nrows) *reinterpret_cast<float4*>(row0 + rr * ld + c * 4) = w;
  }
  __syncwarp();
}

// q/k head of HD columns: bias, RMSNorm with gain g, adjacent-pair RoPE at
// table row `tok`, bf16 store of the whole head row.  Two passes over the
// accumulator (TMEM reads are cheap): the first sums squares, the second
// normalises, rotates and stores 32 columns at a time, so a thread never
// holds more than one 32-column chunk.
template <int HD>
__device__ __forceinline__ void epi_qk_head(uint32_t taddr, const GemmParams& p, int n, const float* __restrict__ g,
                                            int tok, uint8_t* stg, int lane, uint16_t* row0, long long ld,
                                            int nrows, float rs) {
  float ss = 0.f;
#pragma unroll 1
  for (int c = 0; c < HD / 32; ++c) {
    float v[32];
    acc_chunk(taddr + c * 32, p, n + c * 32, v, rs);
#pragma unroll
    for (int i = 0; i < 32; ++i) ss = fmaf(v[i], v[i], ss);
  }
  const float rinv = rsqrtf(ss * (1.0f / HD) + p.eps);
#pragma unroll 1
  for (int c = 0; c < HD / 32; ++c) {
    float v[32];
    acc_chunk(taddr + c * 32, p, n + c * 32, v, rs);
    // pairs 16c .. 16c + 15 of the head: table columns of this token
    const float4* cs4 = reinterpret_cast<const float4*>(p.rope_cos + (long long)tok * (HD / 2) + 16 * c);
    const float4* sn4 = reinterpret_cast<const float4*>(p.rope_sin + (long long)tok * (HD / 2) + 16 * c);
    const float4* g4 = reinterpret_cast<const float4*>(g + 32 * c);
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // 8 channels = 4 pairs per iteration
      const float4 cq = __ldg(cs4 + q);
      const float4 sq = __ldg(sn4 + q);
      const float4 ga = __ldg(g4 + 2 * q);
      const float4 gb = __ldg(g4 + 2 * q + 1);
      const float cc[4] = {cq.x, cq.y, cq.z, cq.w};
      const float sc[4] = {sq.x, sq.y, sq.z, sq.w};
      const float gg[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float x0 = v[8 * q + 2 * j] * rinv * gg[2 * j];
        const float x1 = v[8 * q + 2 * j + 1] * rinv * gg[2 * j + 1];
        v[8 * q + 2 * j] = x0 * cc[j] - x1 * sc[j];
        v[8 * q + 2 * j + 1] = x0 * sc[j] + x1 * cc[j];
      }
    }
    warp_store_bf16x32(stg, lane, v, row0 + 32 * c, ld, nrows);
  }
}

// One epilogue warp's share of a finished 128 x 256 accumulator: the 32 rows
// of its TMEM lane quadrant (thread = row r of the tile) and the 128 columns
// of column half `half`.  `tbase` addresses the quadrant's lanes at column 0
// of the accumulator.
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, const CUtensorMap* tmR, const TileCoord& c,
                                              uint32_t tbase, int r, int half, uint8_t* stg) {
  constexpr int kHalf = kBN / 2;
  const int lane = r & 31;
  const int m = c.tm * kBM + r;
  const int wm0 = m - lane;                                // the warp's first row
  const int nrows = min(32, p.M_seg - wm0);                // rows of this warp inside the problem (may be <= 0)
  const long long orow0 = (long long)c.seg * p.out_seg_rows + p.out_row_off + wm0;
  const int n0 = c.tn * kBN + half * kHalf;                // first output column of this half
  const uint32_t tb = tbase + half * kHalf;
  // fp8 GEMM: this row's activation scale (rows past the problem use 1; they are not stored)
  const float rs = p.ascale && m < p.M_seg ? __ldg(p.ascale + (long long)c.seg * p.ascale_seg_rows + m) : 1.0f;

  if (p.mode == GM_QKV) {
    const int D = p.qkv_D;
    if (n0 < 2 * D) {
      const float* g = n0 < D ? p.gq : p.gk;
      // table row of this token; rows past the problem read row 0 (not stored)
      const int tok = m < p.M_seg ? p.out_row_off + m : 0;
      uint16_t* row0 = p.qk + orow0 * p.qk_ld + n0;
      if (p.d_head == 128) {
        epi_qk_head<128>(tb, p, n0, g, tok, stg, lane, row0, p.qk_ld, nrows, rs);
      } else {
#pragma unroll 1
        for (int h = 0; h < kHalf / 64; ++h)
          epi_qk_head<64>(tb + h * 64, p, n0 + h * 64, g, tok, stg, lane, row0 + h * 64, p.qk_ld, nrows, rs);
      }
    } else if (n0 < 3 * D) {
      // v^T: for each channel, the 32 lanes write 32 consecutive tokens (64 bytes)
      const int tok = p.out_row_off + m;
      uint16_t* vt = p.vT + (long long)c.seg * D * p.vT_ld + tok;
#pragma unroll 1
      for (int j = 0; j < kHalf / 32; ++j) {
        const int n = n0 + j * 32;
        float v[32];
        acc_chunk(tb + j * 32, p, n, v, rs);
        if (lane < nrows) {
          const long long col = n - 2 * D;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            __nv_bfloat16 b = __float2bfloat16_rn(v[i]);
            vt[(col + i) * p.vT_ld] = *reinterpret_cast<uint16_t*>(&b);
          }
        }
      }
    } else {
      uint16_t* row0 = p.aux + orow0 * p.aux_ld + p.aux_col_off - 3 * D;
#pragma unroll 1
      for (int j = 0; j < kHalf / 32; ++j) {
        const int n = n0 + j * 32;
        if (n >= p.N) break;
        float v[32];
        acc_chunk(tb + j * 32, p, n, v, rs);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = gelu_tanh_f(v[i]);
        warp_store_bf16x32(stg, lane, v, row0 + n, p.aux_ld, nrows);
      }
    }
    return;
  }

  if (p.mode == GM_SWIGLU) {
    // accumulator columns [0, 128): gate rows g0 + c; [128, 256): up rows p.swiglu_up + g0 + c.
    // Half h takes gate / up column pairs 64 h .. 64 h + 63.
    const int g0 = c.tn * kHalf;
    uint16_t* row0 = reinterpret_cast<uint16_t*>(p.out) + orow0 * p.out_ld + g0;
#pragma unroll 1
    for (int jj = 0; jj < kHalf / 64; ++jj) {
      const int j = half * (kHalf / 64) + jj;
      float gt[32], u[32];
      acc_chunk(tbase + j * 32, p, g0 + j * 32, gt, rs);
      acc_chunk(tbase + kHalf + j * 32, p, p.swiglu_up + g0 + j * 32, u, rs);
#pragma unroll
      for (int i = 0; i < 32; ++i) gt[i] = silu_fast(gt[i]) * u[i];
      warp_store_bf16x32(stg, lane, gt, row0 + j * 32, p.out_ld, nrows);
    }
    return;
  }

#pragma unroll 1
  for (int j = 0; j < kHalf / 32; ++j) {
    const int n = n0 + j * 32;
    if (n >= p.N) break;
    float v[32];
    acc_chunk(tb + j * 32, p, n, v, rs);
    if (p.mode == GM_STORE_BF16) {
      if (n >= p.gelu_from) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = gelu_tanh_f(v[i]);
      }
      warp_store_bf16x32(stg, lane, v, reinterpret_cast<uint16_t*>(p.out) + orow0 * p.out_ld + n, p.out_ld, nrows);
    } else if (p.mode == GM_STORE_F32) {
      warp_store_f32x32(stg, lane, v, reinterpret_cast<float*>(p.out) + orow0 * p.out_ld + n, p.out_ld, nrows);
    } else {  // GM_RESID: x += gate * v, added in L2 by a TMA reduce-add
      if (p.gate) {
        float gt[32];
        load_vec32(p.gate + (long long)c.seg * p.gate_seg_stride + n, gt);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= gt[i];
      }
      // The warp's 32 rows x 32 columns in the 128-byte-swizzled box layout
      // of the residual's tensor map: row `lane` at a 128-byte pitch, 16-byte
      // chunk j at position j ^ (lane % 8).  The block is reused once the
      // previous reduce has read it.
      if (lane == 0) bulk_wait_group_read0();
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<float4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) =
            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && nrows > 0) {
        tma_reduce_add_3d(tmR, smem_u32(stg), n, wm0, c.seg);
        bulk_commit_group();
      }
    }
  }
}

// F8: A and W are e4m3 (one byte per element, 128 elements per 128-byte
// K slice, kind::f8f6f4 MMAs of K = 32); otherwise bf16 (64 per K slice,
// kind::f16 MMAs of K = 16).  Either way a K slice holds 16 KB of A and
// 16 KB of W per CTA and takes four pair MMAs; a stage holds two slices.
template <bool F8>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_bf16_tc_kernel(const __grid_constant__ GemmGroup g) {
  constexpr int kSL = F8 ? 128 : kBK;  // K elements per slice (one 128-byte row)
  constexpr int kKB = 2 * kSL;         // K elements per stage
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kRing * kStageA;
  // epilogue staging blocks, 4 KB per epilogue warp, on 1024-byte boundaries
  // (the 128-byte swizzle of a TMA copy follows the shared-memory address)
  uint8_t* sE = sB + kRing * kStageB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sE + kEpiWarps * kEpiStageBytes);
  // full[kRing], tempty[2], mma_done: used in CTA 0 only; empty[kRing], tfull[2]: in both CTAs
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + kRing);
  const uint32_t tfull0 = smem_u32(bars + 2 * kRing);
  const uint32_t tempty0 = smem_u32(bars + 2 * kRing + 2);
  const uint32_t mma_done = smem_u32(bars + 2 * kRing + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kRing + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* peer_fills = reinterpret_cast<volatile int*>(tmem_slot + 2);  // CTA 0: CTA 1's fill count

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = (int)cluster_ctarank();
  const int cluster = blockIdx.x >> 1;
  const int n_clusters = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRing; ++s) {
      mbar_init(full0 + 8 * s, 2);  // one arrive.expect_tx from each CTA's producer
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 2 * kEpiWarps);  // the epilogue warps of both CTAs
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    *peer_fills = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int q = 0; q < g.n_prob; ++q) {
      tma_prefetch_desc(&g.tmA[q]);
      tma_prefetch_desc(&g.tmB[q]);
    }
  }
  uint32_t elected = 0;
  if (warp == 1) {
    elected = elect_one_sync();
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  // Both CTAs' barriers are initialised before either CTA's loads, arrivals
  // or commits can reach them.
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  unsigned* const status = g.p[0].status;
  int n_fill = 0;  // stages this CTA's producer has filled (for the drain on exit)

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t full_c0 = mapa_shared(full0, 0);    // CTA 0's full barriers, as seen from this CTA
      int stage = 0;
      uint32_t phase = 0;
      for (int t = cluster; t < g.total_tiles; t += n_clusters) {
        const int q = t < g.tiles0 ? 0 : 1;
        const GemmParams& p = g.p[q];
        const TileCoord c = tile_coord(p, t - (q ? g.tiles0 : 0), rank);
        const int m0 = c.tm * kBM, n0 = c.tn * kBN;
        // W rows of this CTA's half of the 256-row tile: rows n0 + 128 rank, or
        // for SwiGLU the matching 128 gate rows (rank 0) and up rows (rank 1)
        const int brow = p.mode == GM_SWIGLU ? c.tn * (kBN / 2) + rank * p.swiglu_up : n0 + rank * (kBN / 2);
        const int nk = (p.K + kKB - 1) / kKB;
        for (int kb = 0; kb < nk; ++kb) {
          const int ns = p.K - kb * kKB >= kKB ? 2 : 1;  // K slices in this stage
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, status, ST_TIMEOUT_PRODUCER)) goto done;
          const uint32_t fb = full_c0 + 8 * stage;
          if (rank == 0)
            mbar_expect_tx(full0 + 8 * stage, ns * (kHalfA + kHalfB));
          else
            mbar_arrive_expect_tx_cluster(fb, ns * (kHalfA + kHalfB));
          for (int sl = 0; sl < ns; ++sl) {
            tma_load_3d_pair(smem_u32(sA + stage * kStageA + sl * kHalfA), &g.tmA[q], fb, kb * kKB + sl * kSL, m0,
                             c.seg);
            tma_load_3d_pair(smem_u32(sB + stage * kStageB + sl * kHalfB), &g.tmB[q], fb, kb * kKB + sl * kSL, brow, 0);
          }
          ++n_fill;
          if (++stage == kRing) stage = 0, phase ^= 1;
        }
      }
    }
  } else if (warp == 1) {
    if (rank == 0) {
      // The whole warp runs the issue loop (warp-uniform operands); the
      // elected lane issues the pair MMAs and commits.  Descriptors are
      // built once; per MMA only a compile-time offset (in 16-byte units of
      // the start-address field) is added.  The same shared-memory offsets
      // address the operands in both CTAs.
      const uint32_t idesc = F8 ? idesc_e4m3(2 * kBM, kBN) : idesc_bf16(2 * kBM, kBN);
      const uint64_t dA0 = sdesc_k128(smem_u32(sA)), dB0 = sdesc_k128(smem_u32(sB));
      const uint32_t tfull_c1 = mapa_shared(tfull0, 1);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      // Stages this CTA pair fills in all (n_total) and has consumed (n_cons).
      int n_total = 0, n_cons = 0;
      for (int t = cluster; t < g.total_tiles; t += n_clusters) n_total += (g.p[t < g.tiles0 ? 0 : 1].K + kKB - 1) / kKB;
      for (int t = cluster; t < g.total_tiles; t += n_clusters) {
        const int K = g.p[t < g.tiles0 ? 0 : 1].K;
        const int nk = (K + kKB - 1) / kKB;
        if (!mbar_wait_warp(tempty0 + 8 * acc, acc_phase ^ 1, abort_flag, status, ST_TIMEOUT_MMA)) goto done;
        tc_fence_after();
        const uint32_t d = tmem + acc * kBN;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_warp(full0 + 8 * stage, phase, abort_flag, status, ST_TIMEOUT_MMA)) goto done;
          tc_fence_after();
          const int ns = K - kb * kKB >= kKB ? 2 : 1;
#pragma unroll
          for (int sl = 0; sl < 2; ++sl) {
            if (sl < ns) {
              const uint64_t da = dA0 + (uint64_t)((stage * kStageA + sl * kHalfA) >> 4);
              const uint64_t db = dB0 + (uint64_t)((stage * kStageB + sl * kHalfB) >> 4);
#pragma unroll
              for (int k = 0; k < 4; ++k) {  // 32 bytes of K per MMA
                if (F8)
                  umma_f8_pair_if(elected, d, da + 2 * k, db + 2 * k, idesc, (kb | sl | k) != 0);
                else
                  umma_bf16_pair_if(elected, d, da + 2 * k, db + 2 * k, idesc, (kb | sl | k) != 0);
              }
            }
          }
          // One commit frees the stage in both CTAs (multicast to the empty
          // barrier at the same offset in each).  The releases of the last
          // ring round, which no fill waits for, go to CTA 0 only: every
          // arrival that reaches CTA 1 is then one its producer waits for
          // before it leaves the loop, so none can land after CTA 1 exits.
          // (Forwarding each release to CTA 1 through CTA 0's producer made
          // CTA 1's refills later and the K-heavy launches 1.5-2 % slower.)
          if (n_cons + kRing < n_total)
            umma_commit_pair_mc_if(elected, empty0 + 8 * stage, 3);
          else
            umma_commit_pair_if(elected, empty0 + 8 * stage);
          ++n_cons;
          if (++stage == kRing) stage = 0, phase ^= 1;
        }
        umma_commit_pair_if(elected, tfull0 + 8 * acc);
        umma_commit_pair_if(elected, tfull_c1 + 8 * acc);
        if (++acc == 2) acc = 0, acc_phase ^= 1;
      }
    }
  } else {
    // warps 2..9: TMEM lane quadrant warp % 4 (a warp may only read its own
    // quadrant's lanes), column half 0 for warps 2-5 and 1 for warps 6-9
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quad * 32 + lane;
    uint8_t* stg = sE + (warp - 2) * kEpiStageBytes;
    const uint32_t tempty_c0 = mapa_shared(tempty0, 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = cluster; t < g.total_tiles; t += n_clusters) {
      const int q = t < g.tiles0 ? 0 : 1;
      const GemmParams& p = g.p[q];
      const TileCoord c = tile_coord(p, t - (q ? g.tiles0 : 0), rank);
      if (!mbar_wait(tfull0 + 8 * acc, acc_phase, abort_flag, status, ST_TIMEOUT_EPILOGUE)) break;
      tc_fence_after();
      if (c.valid) epilogue_tile(p, &g.tmR[q], c, tmem + ((uint32_t)(quad * 32) << 16) + acc * kBN, r, half, stg);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_c0 + 8 * acc);
      if (++acc == 2) acc = 0, acc_phase ^= 1;
    }
    // this warp's residual reduce-adds have completed (their staging block
    // read, their sums in global memory) before the CTA moves on
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }
done:
  __syncwarp();
  // Every pair MMA of CTA 0 has completed (they read both CTAs' shared
  // memory and write both CTAs' tensor memory) before either CTA moves on.
  if (warp == 1 && rank == 0) {
    umma_commit_pair_if(elected, mma_done);
    mbar_wait_warp(mma_done, 0, nullptr, nullptr, 0);
  }
  // CTA 1 tells CTA 0 how many stages it filled.
  if (warp == 0 && lane == 0 && rank == 1) st_shared_cluster_u32(mapa_shared(smem_u32((const void*)peer_fills), 0), n_fill);
  tc_fence_before();
  cluster_sync();
  if (warp == 0 && lane == 0 && rank == 0) {
    // Every fill of either CTA completes on CTA 0's full barriers.  After a
    // time-out the two producers may have stopped at different fills (at
    // most one ring apart): CTA 0 supplies the arrivals of the CTA that did
    // not fill a stage, then waits (bounded) until the last ring round of
    // fills has landed, so no copy is still writing into either CTA's
    // shared memory when the CTAs exit.  Without a time-out both counts
    // are equal and every wait returns at once.
    const int n_other = *peer_fills;
    const int n_lo = min(n_fill, n_other), n_hi = max(n_fill, n_other);
    for (int i = n_lo; i < n_hi; ++i) {
      if (i >= kRing)
        mbar_wait(full0 + 8 * ((i - kRing) % kRing), (uint32_t)((i - kRing) / kRing) & 1, nullptr, nullptr, 0,
                  100000000ull);
      mbar_arrive(full0 + 8 * (i % kRing));
    }
    for (int i = max(0, n_hi - kRing); i < n_hi; ++i)
      mbar_wait(full0 + 8 * (i % kRing), (uint32_t)(i / kRing) & 1, nullptr, nullptr, 0, 100000000ull);
  }
  __syncwarp();
  // Neither CTA leaves (or frees its tensor memory) before the other is done
  // with its barriers and shared memory.
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_gemm(const GemmGroup& g, cudaStream_t s) {
  // One-time set-up per device (shared-memory opt-in, resident cluster
  // count), safe under concurrent first calls from several host threads.
  static std::once_flag once[64];
  static cudaError_t setup_err[64];
  static int max_clusters[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = kGemmSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  std::call_once(once[dev], [&] {
    cudaError_t e =
        cudaFuncSetAttribute(gemm_bf16_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_bf16_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmem);
    int n = 0;
    if (e == cudaSuccess) {
      // Clusters of two that fit on the device at once (one CTA per SM).
      cudaLaunchConfig_t q = cfg;
      q.gridDim = dim3(2 * (num_sms() / 2));
      e = cudaOccupancyMaxActiveClusters(&n, gemm_bf16_tc_kernel<false>, &q);
    }
    if (e == cudaSuccess && n < 1) e = cudaErrorInvalidConfiguration;
    max_clusters[dev] = n;
    setup_err[dev] = e;
  });
  if (setup_err[dev] != cudaSuccess) return setup_err[dev];
  const int clusters = g.total_tiles < max_clusters[dev] ? g.total_tiles : max_clusters[dev];
  cfg.gridDim = dim3(2 * clusters);
  launch_begin(KID_GEMM, s);
  cudaError_t e = g.f8 ? cudaLaunchKernelEx(&cfg, gemm_bf16_tc_kernel<true>, g)
                       : cudaLaunchKernelEx(&cfg, gemm_bf16_tc_kernel<false>, g);
  launch_end(s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mmdit
