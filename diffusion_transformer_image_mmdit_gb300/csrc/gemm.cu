// Persistent tcgen05 GEMM for the block linears: Y = X W^T with fused epilogues.
//
// The linears of both block types (QKV, output projection, MLP in/out, the
// single block's fused D -> 3D + D_mlp and its 5D -> D output) are dense
// bf16 contractions with fp32 accumulation (Luminal blog, section "The AMD
// MI300X pipeline": all bf16 GEMMs accumulate in fp32, with bias epilogues).
//
// Structure (one CTA per SM, 192 threads):
//   warp 0      TMA producer: A tile 128x64 and B tile 256x64 per K block
//               into a 4-stage ring (128-byte swizzle).
//   warp 1      allocates 512 TMEM columns (two 128x256 fp32 accumulators)
//               and issues tcgen05.mma (M=128, N=256, K=16) from one thread.
//   warps 2-5   epilogue: tcgen05.ld of the finished accumulator (one TMEM
//               lane = one output row per thread), fused bias / per-channel
//               int8 scale / GELU-tanh / gated fp32 residual / q-k RMSNorm +
//               RoPE / transposed V store, overlapping the next tile's MMAs.
#include "common.cuh"

namespace mmdit {

namespace {

constexpr int kGemmThreads = 192;
constexpr uint32_t kStageA = kBM * kBK * 2;  // 16 KB
constexpr uint32_t kStageB = kBN * kBK * 2;  // 32 KB
constexpr uint32_t kTmemCols = 512;
constexpr size_t kGemmSmem = 1024 + kStages * (kStageA + kStageB) + 256;

struct TileCoord {
  int seg, tm, tn;
};

// Grouped raster: runs of group_m M tiles (over all segments) sweep all N
// tiles with M fastest, so the CTAs of one wave share A and B tiles in L2.
__device__ __forceinline__ TileCoord tile_coord(const GemmParams& p, int t) {
  const int total_m = p.n_seg * p.tiles_m;
  const int per_group = p.group_m * p.tiles_n;
  const int g = t / per_group;
  const int first_m = g * p.group_m;
  const int gm = min(p.group_m, total_m - first_m);
  const int r = t - g * per_group;
  const int mi = first_m + r % gm;
  TileCoord c;
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

// Reads 32 accumulator columns of this thread's row and applies the int8
// scale and the bias.
__device__ __forceinline__ void acc_chunk(uint32_t taddr, const GemmParams& p, int n, float* v) {
  uint32_t raw[32];
  MMDIT_TMEM_LD32(taddr, raw);
  tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(raw[i]);
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

__device__ __forceinline__ void store_bf16x32(uint16_t* dst, const float* v) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
    w.y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
    w.z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
    w.w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
    d4[i] = w;
  }
}

// q/k head of HD columns: bias, RMSNorm with gain g, adjacent-pair RoPE at
// table row `tok`, bf16 store of the whole head row.
template <int HD>
__device__ __forceinline__ void epi_qk_head(uint32_t taddr, const GemmParams& p, int n, const float* __restrict__ g,
                                            int tok, bool valid, uint16_t* dst) {
  float v[HD];
#pragma unroll
  for (int c = 0; c < HD / 32; ++c) acc_chunk(taddr + c * 32, p, n + c * 32, v + c * 32);
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < HD; ++i) ss = fmaf(v[i], v[i], ss);
  const float rs = rsqrtf(ss * (1.0f / HD) + p.eps);
  if (!valid) return;
  const float4* cs4 = reinterpret_cast<const float4*>(p.rope_cos + (long long)tok * (HD / 2));
  const float4* sn4 = reinterpret_cast<const float4*>(p.rope_sin + (long long)tok * (HD / 2));
  const float4* g4 = reinterpret_cast<const float4*>(g);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < HD / 8; ++q) {  // 8 channels = 4 pairs per iteration
    const float4 c = __ldg(cs4 + q);
    const float4 s = __ldg(sn4 + q);
    const float4 ga = __ldg(g4 + 2 * q);
    const float4 gb = __ldg(g4 + 2 * q + 1);
    const float cc[4] = {c.x, c.y, c.z, c.w};
    const float sc[4] = {s.x, s.y, s.z, s.w};
    const float gg[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float x0 = v[8 * q + 2 * j] * rs * gg[2 * j];
      const float x1 = v[8 * q + 2 * j + 1] * rs * gg[2 * j + 1];
      w[j] = pack_bf16x2(x0 * cc[j] - x1 * sc[j], x0 * sc[j] + x1 * cc[j]);
    }
    d4[q] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

__device__ __forceinline__ void epilogue_tile(const GemmParams& p, const TileCoord& c, uint32_t tbase, int r) {
  const int m = c.tm * kBM + r;
  const bool valid = m < p.M_seg;
  const long long orow = (long long)c.seg * p.out_seg_rows + p.out_row_off + m;
  const int n0 = c.tn * kBN;

  if (p.mode == GM_QKV) {
    const int D = p.qkv_D;
    const int tok = p.out_row_off + m;
    if (n0 < 2 * D) {
      const float* g = n0 < D ? p.gq : p.gk;
      uint16_t* dst = p.qk + orow * p.qk_ld;
      if (p.d_head == 128) {
#pragma unroll 1
        for (int h = 0; h < kBN / 128; ++h)
          epi_qk_head<128>(tbase + h * 128, p, n0 + h * 128, g, tok, valid, dst + n0 + h * 128);
      } else {
#pragma unroll 1
        for (int h = 0; h < kBN / 64; ++h)
          epi_qk_head<64>(tbase + h * 64, p, n0 + h * 64, g, tok, valid, dst + n0 + h * 64);
      }
    } else if (n0 < 3 * D) {
      uint16_t* vt = p.vT + (long long)c.seg * D * p.vT_ld + tok;
#pragma unroll 1
      for (int j = 0; j < kBN / 32; ++j) {
        const int n = n0 + j * 32;
        float v[32];
        acc_chunk(tbase + j * 32, p, n, v);
        if (valid) {
          const long long col = n - 2 * D;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            __nv_bfloat16 b = __float2bfloat16_rn(v[i]);
            vt[(col + i) * p.vT_ld] = *reinterpret_cast<uint16_t*>(&b);
          }
        }
      }
    } else {
      uint16_t* dst = p.aux + orow * p.aux_ld + p.aux_col_off - 3 * D;
#pragma unroll 1
      for (int j = 0; j < kBN / 32; ++j) {
        const int n = n0 + j * 32;
        if (n >= p.N) break;
        float v[32];
        acc_chunk(tbase + j * 32, p, n, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = gelu_tanh_f(v[i]);
        if (valid) store_bf16x32(dst + n, v);
      }
    }
    return;
  }

#pragma unroll 1
  for (int j = 0; j < kBN / 32; ++j) {
    const int n = n0 + j * 32;
    if (n >= p.N) break;
    float v[32];
    acc_chunk(tbase + j * 32, p, n, v);
    if (p.mode == GM_STORE_BF16) {
      if (n >= p.gelu_from) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = gelu_tanh_f(v[i]);
      }
      if (valid) store_bf16x32(reinterpret_cast<uint16_t*>(p.out) + orow * p.out_ld + n, v);
    } else if (p.mode == GM_STORE_F32) {
      if (valid) {
        float4* d4 = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + orow * p.out_ld + n);
#pragma unroll
        for (int i = 0; i < 8; ++i) d4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      }
    } else {  // GM_RESID
      float gt[32];
      if (p.gate) {
        load_vec32(p.gate + (long long)c.seg * p.gate_seg_stride + n, gt);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) gt[i] = 1.0f;
      }
      if (valid) {
        float4* x4 = reinterpret_cast<float4*>(p.resid + ((long long)c.seg * p.resid_seg_rows + m) * p.resid_ld + n);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float4 x = x4[i];
          x.x = fmaf(gt[4 * i], v[4 * i], x.x);
          x.y = fmaf(gt[4 * i + 1], v[4 * i + 1], x.y);
          x.z = fmaf(gt[4 * i + 2], v[4 * i + 2], x.z);
          x.w = fmaf(gt[4 * i + 3], v[4 * i + 3], x.w);
          x4[i] = x;
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kGemmThreads, 1) gemm_bf16_tc_kernel(const __grid_constant__ GemmGroup g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kStageA;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kStages * kStageB);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + kStages);
  const uint32_t tfull0 = smem_u32(bars + 2 * kStages);
  const uint32_t tempty0 = smem_u32(bars + 2 * kStages + 2);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 4);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int q = 0; q < g.n_prob; ++q) {
      tma_prefetch_desc(&g.tmA[q]);
      tma_prefetch_desc(&g.tmB[q]);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  unsigned* const status = g.p[0].status;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int t = blockIdx.x; t < g.total_tiles; t += gridDim.x) {
        const int q = t < g.tiles0 ? 0 : 1;
        const GemmParams& p = g.p[q];
        const TileCoord c = tile_coord(p, t - (q ? g.tiles0 : 0));
        const int m0 = c.tm * kBM, n0 = c.tn * kBN;
        const int nk = p.K / kBK;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, status, ST_TIMEOUT_PRODUCER)) goto done;
          mbar_expect_tx(full0 + 8 * stage, kStageA + kStageB);
          tma_load_3d(smem_u32(sA + stage * kStageA), &g.tmA[q], full0 + 8 * stage, kb * kBK, m0, c.seg);
          tma_load_3d(smem_u32(sB + stage * kStageB), &g.tmB[q], full0 + 8 * stage, kb * kBK, n0, 0);
          if (++stage == kStages) stage = 0, phase ^= 1;
        }
      }
    }
  } else if (warp == 1) {
    // The whole warp runs the issue loop (warp-uniform operands); the
    // elected lane issues the MMAs and commits.  Descriptors are built once;
    // per MMA only a compile-time offset (in 16-byte units of the
    // start-address field) is added.
    const uint32_t leader = elect_one_sync();
    const uint32_t idesc = idesc_bf16(kBM, kBN);
    const uint64_t dA0 = sdesc_k128(smem_u32(sA)), dB0 = sdesc_k128(smem_u32(sB));
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < g.total_tiles; t += gridDim.x) {
      const int nk = g.p[t < g.tiles0 ? 0 : 1].K / kBK;
      if (!mbar_wait_warp(tempty0 + 8 * acc, acc_phase ^ 1, abort_flag, status, ST_TIMEOUT_MMA)) goto done;
      tc_fence_after();
      const uint32_t d = tmem + acc * kBN;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait_warp(full0 + 8 * stage, phase, abort_flag, status, ST_TIMEOUT_MMA)) goto done;
        tc_fence_after();
        const uint64_t da = dA0 + (uint64_t)(stage * (kStageA >> 4));
        const uint64_t db = dB0 + (uint64_t)(stage * (kStageB >> 4));
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) umma_bf16_if(leader, d, da + 2 * k, db + 2 * k, idesc, (kb | k) != 0);
        umma_commit_if(leader, empty0 + 8 * stage);
        if (++stage == kStages) stage = 0, phase ^= 1;
      }
      umma_commit_if(leader, tfull0 + 8 * acc);
      if (++acc == 2) acc = 0, acc_phase ^= 1;
    }
  } else {
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < g.total_tiles; t += gridDim.x) {
      const int q = t < g.tiles0 ? 0 : 1;
      const GemmParams& p = g.p[q];
      const TileCoord c = tile_coord(p, t - (q ? g.tiles0 : 0));
      if (!mbar_wait(tfull0 + 8 * acc, acc_phase, abort_flag, status, ST_TIMEOUT_EPILOGUE)) break;
      tc_fence_after();
      epilogue_tile(p, c, tmem + ((uint32_t)(quad * 32) << 16) + acc * kBN, r);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
      if (++acc == 2) acc = 0, acc_phase ^= 1;
    }
  }
done:
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_gemm(const GemmGroup& g, cudaStream_t s) {
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(gemm_bf16_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int grid = g.total_tiles < num_sms() ? g.total_tiles : num_sms();
  launch_begin(KID_GEMM, s);
  gemm_bf16_tc_kernel<<<grid, kGemmThreads, kGemmSmem, s>>>(g);
  launch_end(s);
  return cudaGetLastError();
}

}  // namespace mmdit
