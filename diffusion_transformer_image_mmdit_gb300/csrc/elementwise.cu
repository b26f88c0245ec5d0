// Bandwidth-bound kernels of the step: LayerNorm + adaLN modulate, the
// modulation / timestep GEMVs, RoPE tables and rotation, the Euler update,
// the int8 quantiser and dequantiser, and the attention input prep.
// Vectorised 16-byte global accesses, one warp per row where a row reduces.
#include <mutex>

#include "common.cuh"
#include "elementwise.h"

namespace mmdit {

namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Two fp32 values to e4m3 (round to nearest even, saturating at +-448); lo in
// the low byte.
__device__ __forceinline__ uint16_t f8x2_e4m3(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// ------------------------------------------------------------------ LN + modulate
// y = (x - mean) / sqrt(var + eps) * (1 + scale) + shift over one row of D
// floats per warp: lane l holds the float4 chunks l, l + 32, ... (NV = D/128
// of them), so both statistics reduce with shuffles alone (no block
// barrier), and the row stays in registers between the two passes.  fp32
// statistics, the variance from the centred values.
//
// One launch serves up to two jobs (the text and image streams of a double
// block at one LN position): warp rows [0, n0) belong to job 0, the rest to
// job 1, so no launch is as short as one stream's text rows.
//
// F8: the row is also quantised to e4m3 the way the standalone row quantiser
// does it from the stored bf16 values: s = max|bf16(y)| / 448 (1 for a zero
// row), q = e4m3(bf16(y) / s), written to q (row stride D) and qs; the bf16
// row is stored only when y is given.
template <int NV, bool F8>
__global__ void __launch_bounds__(128) ln_mod_kernel(const __grid_constant__ LnJobs J) {
  constexpr int D = NV * 128;
  const int grow = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (grow >= J.n_total) return;
  const int jb = grow < J.n0 ? 0 : 1;
  const LnJob& jo = J.job[jb];
  const int row = grow - (jb ? J.n0 : 0);  // row of this job (output row)
  const int seg = row / jo.rows, i = row - seg * jo.rows;
  const float4* xr = reinterpret_cast<const float4*>(jo.x + ((long long)seg * jo.x_seg_rows + i) * D) + lane;
  float4 v[NV];
#pragma unroll
  for (int c = 0; c < NV; ++c) v[c] = __ldg(xr + 32 * c);
  constexpr float inv_d = 1.0f / (float)D;
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < NV; ++c) s += (v[c].x + v[c].y) + (v[c].z + v[c].w);
  const float mean = warp_sum(s) * inv_d;
  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < NV; ++c) {
    v[c].x -= mean, v[c].y -= mean, v[c].z -= mean, v[c].w -= mean;
    ss = fmaf(v[c].x, v[c].x, fmaf(v[c].y, v[c].y, fmaf(v[c].z, v[c].z, fmaf(v[c].w, v[c].w, ss))));
  }
  const float rstd = rsqrtf(warp_sum(ss) * inv_d + J.eps);
  const float4* sc4 = reinterpret_cast<const float4*>(jo.scale + (long long)seg * jo.mod_stride) + lane;
  const float4* sh4 = reinterpret_cast<const float4*>(jo.shift + (long long)seg * jo.mod_stride) + lane;
  uint2* yr = jo.y ? reinterpret_cast<uint2*>(jo.y + (long long)row * D) + lane : nullptr;
  float amax = 0.f;
#pragma unroll
  for (int c = 0; c < NV; ++c) {
    const float4 sc = __ldg(sc4 + 32 * c), sh = __ldg(sh4 + 32 * c);
    const uint2 o = make_uint2(pack_bf16x2(v[c].x * rstd * (1.f + sc.x) + sh.x, v[c].y * rstd * (1.f + sc.y) + sh.y),
                               pack_bf16x2(v[c].z * rstd * (1.f + sc.z) + sh.z, v[c].w * rstd * (1.f + sc.w) + sh.w));
    if (!F8 || yr) yr[32 * c] = o;
    if (F8) {
      // keep the bf16-rounded values for the quantisation
      v[c] = make_float4(bf16_lo(o.x), bf16_hi(o.x), bf16_lo(o.y), bf16_hi(o.y));
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[c].x), fabsf(v[c].y)), fmaxf(fabsf(v[c].z), fabsf(v[c].w))));
    }
  }
  if (F8) {
    amax = warp_max(amax);
    const float sq = amax == 0.f ? 1.0f : __fdiv_rn(amax, 448.0f);
    if (lane == 0) jo.qs[row] = sq;
    uint32_t* qr = reinterpret_cast<uint32_t*>(jo.q + (long long)row * D) + lane;
#pragma unroll
    for (int c = 0; c < NV; ++c)
      qr[32 * c] = (uint32_t)f8x2_e4m3(__fdiv_rn(v[c].x, sq), __fdiv_rn(v[c].y, sq)) |
                   ((uint32_t)f8x2_e4m3(__fdiv_rn(v[c].z, sq), __fdiv_rn(v[c].w, sq)) << 16);
  }
}

// ------------------------------------------------------------------ sequence-parallel exchange layouts
// Ulysses sequence parallelism swaps a token shard with all heads for all
// tokens with a head group.  pack: src rows [rows][src_ld] hold `sections`
// consecutive sections (q | k | v) of `groups` head groups of gc columns
// each; dst [groups][rows][sections][gc], so that the chunk for head group g
// is contiguous.  unpack: src [groups][rows][gc] -> dst [rows][dst_ld] at
// columns g * gc + c.  A CTA moves whole rows (grid-stride over rows), its
// threads striding over the row's 16-byte vectors (8 bf16): the source row
// is read contiguously, and every run of gc / 8 vectors lands contiguously.
// Index arithmetic in 32 bits per row (one row holds at most 2^31 vectors).
__global__ void __launch_bounds__(256) heads_pack_kernel(const uint16_t* __restrict__ src, long long rows, int src_ld,
                                                         int sections, int groups, int gc,
                                                         uint16_t* __restrict__ dst) {
  const int v8 = gc / 8;
  const int per_row = sections * groups * v8;
  for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src + r * src_ld);
    for (int j = threadIdx.x; j < per_row; j += blockDim.x) {
      const int sg = j / v8, c = j - sg * v8;  // source column block sg = sct * groups + g
      const int sct = sg / groups, g = sg - sct * groups;
      const uint4 v = s4[j];
      *reinterpret_cast<uint4*>(dst + (((long long)g * rows + r) * sections + sct) * gc + 8 * c) = v;
    }
  }
}

__global__ void __launch_bounds__(256) heads_unpack_kernel(const uint16_t* __restrict__ src, long long rows,
                                                           int groups, int gc, uint16_t* __restrict__ dst,
                                                           int dst_ld) {
  const int v8 = gc / 8;
  const int per_row = groups * v8;
  for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
    uint4* d4 = reinterpret_cast<uint4*>(dst + r * dst_ld);
    for (int j = threadIdx.x; j < per_row; j += blockDim.x) {
      const int g = j / v8, c = j - g * v8;
      d4[j] = *reinterpret_cast<const uint4*>(src + ((long long)g * rows + r) * gc + 8 * c);
    }
  }
}

// ------------------------------------------------------------------ GEMV
// y[b, n] = sum_k W[n, k] act(x[b, k]) (* scale[n]) + bias[n] for B <= 8 rows
// of x (K a multiple of 16): one warp per output row (for B > 1, per group of
// kGemvRowsPerWarp rows handled together), 16-byte weight loads along K, x
// staged in shared memory after the activation once per CTA.  The grid is a few CTAs
// per SM striding over the rows, so the staging is paid once per CTA rather
// than once per 32 rows.
constexpr int kGemvRowsPerWarp = 4;
constexpr int kGemvWarps = 8;
constexpr int kGemvVecBatch = 12;  // a whole 3072-wide bf16 row per lane in flight
constexpr int kGemvCtasPerSm = 4;

// Shared-memory slot of x[k] in a staged row.  Lane l reads the weights of
// 16-byte vectors v = l, l + 32, ... (EPV = 8 bf16 or 16 int8 values) and, for
// each, the EPV / 4 float4s of x at the same positions.  Stored plainly, the
// float4s of 8 consecutive lanes would sit 32 or 64 bytes apart (2- or 4-way
// bank conflicts); float4 j of vector v is therefore kept at slot
// j ^ sw(v) of the vector, sw(v) = (v >> 2) & 1 (bf16) or (v >> 1) & 3 (int8),
// which spreads any 8 consecutive lanes over 8 distinct bank groups.
template <bool I8>
__device__ __forceinline__ int gemv_slot(int k) {
  constexpr int EPV = I8 ? 16 : 8;
  const int v = k / EPV, j = (k % EPV) >> 2;
  const int sw = I8 ? ((v >> 1) & 3) : ((v >> 2) & 1);
  return v * EPV + 4 * (j ^ sw) + (k & 3);
}

// One output row (K a multiple of EPV): up to kGemvVecBatch 16-byte weight
// loads per lane in flight before use; B <= BM rows of x (BM a compile-time
// bound, so B = 1 keeps one accumulator and few registers).
template <bool I8, int BM>
__device__ __forceinline__ void gemv_row(const uint8_t* __restrict__ wrow, const float* xs, int B, int K, int lane,
                                         float* acc) {
  constexpr int EPV = I8 ? 16 : 8;
  const int nvec = K / EPV;
  const uint4* wr = reinterpret_cast<const uint4*>(wrow);
#pragma unroll 1
  for (int v0 = lane; v0 < nvec; v0 += 32 * kGemvVecBatch) {
    uint4 wv[kGemvVecBatch];
#pragma unroll
    for (int u = 0; u < kGemvVecBatch; ++u)
      if (v0 + 32 * u < nvec) wv[u] = __ldg(wr + v0 + 32 * u);
#pragma unroll
    for (int u = 0; u < kGemvVecBatch; ++u) {
      const int v = v0 + 32 * u;
      if (v >= nvec) break;
      float w[EPV];
      const uint32_t q[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
      if (I8) {
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = (float)(int8_t)((q[e >> 2] >> (8 * (e & 3))) & 0xFF);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) w[2 * e] = bf16_lo(q[e]), w[2 * e + 1] = bf16_hi(q[e]);
      }
      const int sw = I8 ? ((v >> 1) & 3) : ((v >> 2) & 1);
#pragma unroll
      for (int b = 0; b < BM; ++b) {
        if (b < B) {
          const float4* xv = reinterpret_cast<const float4*>(xs + b * K + v * EPV);
          float t = acc[b];
#pragma unroll
          for (int j = 0; j < EPV / 4; ++j) {
            const float4 xj = xv[j ^ sw];
            t = fmaf(w[4 * j + 3], xj.w, fmaf(w[4 * j + 2], xj.z, fmaf(w[4 * j + 1], xj.y, fmaf(w[4 * j], xj.x, t))));
          }
          acc[b] = t;
        }
      }
    }
  }
}

// Four int8 values (one 32-bit word) to fp32, exactly, on the FMA pipe
// instead of four int-to-float conversions: with its sign bit flipped the
// byte b becomes q + 128 in 0..255; placed as the low mantissa byte of the
// float 2^23 it gives 2^23 + q + 128, from which 2^23 + 128 is subtracted.
__device__ __forceinline__ void i8x4_to_f32(uint32_t q, float* w) {
  const uint32_t u = q ^ 0x80808080u;
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540u | i)) - 8388736.0f;
}

// The NR rows of one warp at once, for batches B > 1: the weight vectors at
// one K position are loaded for all NR rows, and the x values there (all B
// rows of x) are read from shared memory once for the NR rows.  One row at a
// time reads B * 4 float4s of x per 16-byte weight vector -- 256 bytes per 16
// weight bytes with B = 4 and int8 weights, which made the kernel bound by
// shared memory; sharing them cuts that NR-fold.  wrow[r] is null for rows
// past the end.
template <bool I8, int BM, int NR>
__device__ __forceinline__ void gemv_rows(const uint8_t* const* wrow, const float* xs, int B, int K, int lane,
                                          float (&acc)[NR][BM]) {
  constexpr int EPV = I8 ? 16 : 8;
  constexpr int U = kGemvVecBatch / NR;  // vectors per row in flight: kGemvVecBatch loads per lane
  const int nvec = K / EPV;
#pragma unroll 1
  for (int v0 = lane; v0 < nvec; v0 += 32 * U) {
    uint4 wv[NR][U];
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (wrow[r] && v0 + 32 * u < nvec) wv[r][u] = __ldg(reinterpret_cast<const uint4*>(wrow[r]) + v0 + 32 * u);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + 32 * u;
      if (v >= nvec) break;
      const int sw = I8 ? ((v >> 1) & 3) : ((v >> 2) & 1);
      // the vector in two halves of EPV / 2 elements, so that only half of
      // its x values (for all B rows) are held at a time
#pragma unroll
      for (int hv = 0; hv < 2; ++hv) {
        constexpr int Q = EPV / 8;  // float4s of x per half vector and row
        float4 xv[BM][Q];
#pragma unroll
        for (int b = 0; b < BM; ++b)
#pragma unroll
          for (int j = 0; j < Q; ++j)
            xv[b][j] = b < B ? reinterpret_cast<const float4*>(xs + b * K + v * EPV)[(hv * Q + j) ^ sw]
                             : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          if (!wrow[r]) continue;
          float w[EPV / 2];
          const uint32_t q0 = hv ? wv[r][u].z : wv[r][u].x, q1 = hv ? wv[r][u].w : wv[r][u].y;
          if (I8) {
            i8x4_to_f32(q0, w);
            i8x4_to_f32(q1, w + 4);
          } else {
            w[0] = bf16_lo(q0), w[1] = bf16_hi(q0), w[2] = bf16_lo(q1), w[3] = bf16_hi(q1);
          }
#pragma unroll
          for (int b = 0; b < BM; ++b) {
            float t = acc[r][b];
#pragma unroll
            for (int j = 0; j < Q; ++j)
              t = fmaf(w[4 * j + 3], xv[b][j].w, fmaf(w[4 * j + 2], xv[b][j].z,
                       fmaf(w[4 * j + 1], xv[b][j].y, fmaf(w[4 * j], xv[b][j].x, t))));
            acc[r][b] = t;
          }
        }
      }
    }
  }
}

template <bool I8>
__device__ __forceinline__ void gemv_stage_x(const float* __restrict__ x, int B, int K, int act, float* xs) {
  for (int i = threadIdx.x; i < B * K; i += blockDim.x) {
    const float t = x[i];
    const int b = i / K, k = i - b * K;
    xs[b * K + gemv_slot<I8>(k)] = act ? silu_f(t) : t;
  }
  __syncthreads();
}


template <bool I8, int BM>
__global__ void __launch_bounds__(256) gemv_kernel(const void* __restrict__ W, const float* __restrict__ wscale,
                                                   const float* __restrict__ bias, const float* __restrict__ x, int B,
                                                   int N, int K, int act, float* __restrict__ y) {
  extern __shared__ float xs[];
  gemv_stage_x<I8>(x, B, K, act, xs);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int stride = gridDim.x * kGemvWarps * kGemvRowsPerWarp;
#pragma unroll 1
  for (int row0 = (blockIdx.x * kGemvWarps + warp) * kGemvRowsPerWarp; row0 < N; row0 += stride) {
#pragma unroll 1
    for (int rr = 0; rr < kGemvRowsPerWarp; ++rr) {
      const int n = row0 + rr;
      if (n >= N) break;
      float acc[BM];
#pragma unroll
      for (int b = 0; b < BM; ++b) acc[b] = 0.f;
      gemv_row<I8, BM>(reinterpret_cast<const uint8_t*>(W) + (long long)n * K * (I8 ? 1 : 2), xs, B, K, lane, acc);
      const float sc = wscale ? wscale[n] : 1.0f;
      const float bi = bias ? bias[n] : 0.0f;
#pragma unroll
      for (int b = 0; b < BM; ++b) {
        if (b < B) {
          const float t = warp_sum(acc[b]);
          if (lane == 0) y[(long long)b * N + n] = t * sc + bi;
        }
      }
    }
  }
}

// Batched form: the jobs' output rows are numbered consecutively; each warp
// finds the job of its row in the kernel-parameter table (its rows only
// increase, so the search resumes where it stopped).
constexpr int kMaxGemvJobs = 96;
struct GemvBatch {
  GemvJob job[kMaxGemvJobs];
  int row0[kMaxGemvJobs + 1];
  int n_jobs;
};

template <bool I8, int BM>
__global__ void __launch_bounds__(256) gemv_batched_kernel(const __grid_constant__ GemvBatch jb,
                                                           const float* __restrict__ x, int B, int K, int act) {
  extern __shared__ float xs[];
  gemv_stage_x<I8>(x, B, K, act, xs);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = jb.row0[jb.n_jobs];
  const int stride = gridDim.x * kGemvWarps * kGemvRowsPerWarp;
  int j = 0;
#pragma unroll 1
  for (int row_base = (blockIdx.x * kGemvWarps + warp) * kGemvRowsPerWarp; row_base < total; row_base += stride) {
#pragma unroll 1
    for (int rr = 0; rr < kGemvRowsPerWarp; ++rr) {
      const int R = row_base + rr;
      if (R >= total) break;
      while (R >= jb.row0[j + 1]) ++j;
      const GemvJob& job = jb.job[j];
      const int n = R - jb.row0[j];
      float acc[BM];
#pragma unroll
      for (int b = 0; b < BM; ++b) acc[b] = 0.f;
      gemv_row<I8, BM>(reinterpret_cast<const uint8_t*>(job.W) + (long long)n * K * (I8 ? 1 : 2), xs, B, K, lane, acc);
      const float sc = job.scale ? job.scale[n] : 1.0f;
      const float bi = job.bias ? job.bias[n] : 0.0f;
#pragma unroll
      for (int b = 0; b < BM; ++b) {
        if (b < B) {
          const float t = warp_sum(acc[b]);
          if (lane == 0) job.out[(long long)b * (job.ldo ? job.ldo : job.N) + n] = t * sc + bi;
        }
      }
    }
  }
}


// B > 1: the same two kernels with the kGemvRowsPerWarp rows of a warp
// handled together (gemv_rows); two CTAs per SM keep enough loads in flight.
template <bool I8, int BM>
__global__ void __launch_bounds__(256, 2) gemv_rows_kernel(const void* __restrict__ W, const float* __restrict__ wscale,
                                                           const float* __restrict__ bias, const float* __restrict__ x,
                                                           int B, int N, int K, int act, float* __restrict__ y) {
  extern __shared__ float xs[];
  gemv_stage_x<I8>(x, B, K, act, xs);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int stride = gridDim.x * kGemvWarps * kGemvRowsPerWarp;
#pragma unroll 1
  for (int row0 = (blockIdx.x * kGemvWarps + warp) * kGemvRowsPerWarp; row0 < N; row0 += stride) {
    const uint8_t* wrow[kGemvRowsPerWarp];
#pragma unroll
    for (int rr = 0; rr < kGemvRowsPerWarp; ++rr)
      wrow[rr] = row0 + rr < N ? reinterpret_cast<const uint8_t*>(W) + (long long)(row0 + rr) * K * (I8 ? 1 : 2)
                               : nullptr;
    float acc[kGemvRowsPerWarp][BM];
#pragma unroll
    for (int rr = 0; rr < kGemvRowsPerWarp; ++rr)
#pragma unroll
      for (int b = 0; b < BM; ++b) acc[rr][b] = 0.f;
    gemv_rows<I8, BM, kGemvRowsPerWarp>(wrow, xs, B, K, lane, acc);
#pragma unroll
    for (int rr = 0; rr < kGemvRowsPerWarp; ++rr) {
      const int n = row0 + rr;
      if (n >= N) break;
      const float sc = wscale ? wscale[n] : 1.0f;
      const float bi = bias ? bias[n] : 0.0f;
#pragma unroll
      for (int b = 0; b < BM; ++b) {
        if (b < B) {
          const float t = warp_sum(acc[rr][b]);
          if (lane == 0) y[(long long)b * N + n] = t * sc + bi;
        }
      }
    }
  }
}

template <bool I8, int BM>
__global__ void __launch_bounds__(256, 2) gemv_rows_batched_kernel(const __grid_constant__ GemvBatch jb,
                                                                   const float* __restrict__ x, int B, int K, int act) {
  extern __shared__ float xs[];
  gemv_stage_x<I8>(x, B, K, act, xs);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = jb.row0[jb.n_jobs];
  const int stride = gridDim.x * kGemvWarps * kGemvRowsPerWarp;
  int j = 0;
#pragma unroll 1
  for (int row_base = (blockIdx.x * kGemvWarps + warp) * kGemvRowsPerWarp; row_base < total; row_base += stride) {
    const uint8_t* wrow[kGemvRowsPerWarp];
    int jr[kGemvRowsPerWarp], nr[kGemvRowsPerWarp];
#pragma unroll
    for (int rr = 0; rr < kGemvRowsPerWarp; ++rr) {
      const int R = row_base + rr;
      wrow[rr] = nullptr;
      jr[rr] = j;
      nr[rr] = 0;
      if (R < total) {
        while (R >= jb.row0[j + 1]) ++j;
        jr[rr] = j;
        nr[rr] = R - jb.row0[j];
        wrow[rr] = reinterpret_cast<const uint8_t*>(jb.job[j].W) + (long long)nr[rr] * K * (I8 ? 1 : 2);
      }
    }
    float acc[kGemvRowsPerWarp][BM];
#pragma unroll
    for (int rr = 0; rr < kGemvRowsPerWarp; ++rr)
#pragma unroll
      for (int b = 0; b < BM; ++b) acc[rr][b] = 0.f;
    gemv_rows<I8, BM, kGemvRowsPerWarp>(wrow, xs, B, K, lane, acc);
#pragma unroll
    for (int rr = 0; rr < kGemvRowsPerWarp; ++rr) {
      if (!wrow[rr]) break;
      const GemvJob& job = jb.job[jr[rr]];
      const int n = nr[rr];
      const float sc = job.scale ? job.scale[n] : 1.0f;
      const float bi = job.bias ? job.bias[n] : 0.0f;
#pragma unroll
      for (int b = 0; b < BM; ++b) {
        if (b < B) {
          const float t = warp_sum(acc[rr][b]);
          if (lane == 0) job.out[(long long)b * (job.ldo ? job.ldo : job.N) + n] = t * sc + bi;
        }
      }
    }
  }
}


// ------------------------------------------------------------------ timestep sinusoid
// t_tab != null: t = t_scale * t_tab[*t_idx] (the step's sigma read on the
// device, so that a captured step replays for every step of a schedule).
__global__ void sinusoid_kernel(double t, const double* __restrict__ t_tab, const int* __restrict__ t_idx,
                                double t_scale, int B, int dim, float* __restrict__ out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int half = dim / 2;
  if (i >= B * dim) return;
  if (t_tab) t = t_scale * t_tab[*t_idx];
  const int j = i % dim;
  const int jj = j < half ? j : j - half;
  const double f = exp(-log(10000.0) * (double)jj / (double)half);
  const double a = t * f;
  out[i] = (float)(j < half ? cos(a) : sin(a));
}

// y[i] += x[i]
__global__ void add_f32_kernel(float* __restrict__ y, const float* __restrict__ x, long long n) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) y[i] += x[i];
}

// dst[i] = src[k * stride + i] for i < n (n, stride multiples of 4, 16-byte
// aligned), with k = *k_dev when given (the device step counter of a replayed
// step), else k_host: one step's slice of buffers computed for every step.
__global__ void select_step_kernel(const float4* __restrict__ src, long long stride4, long long n4,
                                   const int* __restrict__ k_dev, int k_host, float4* __restrict__ dst) {
  const long long k = k_dev ? *k_dev : k_host;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x)
    dst[i] = src[k * stride4 + i];
}

// The device step counter of a replayed step: set once, advanced at the end of each step.
__global__ void counter_kernel(int* c, int value, int add) { *c = add ? *c + value : value; }

// ------------------------------------------------------------------ RoPE
// ids [L,3] and cos/sin [L, d/2]: angle = pos_axis * theta^(-2i/d_axis), fp64,
// rounded once to fp32.  Tokens: L_txt text at (0, 0, 0), then n_gen target
// image tokens at (0, h, w) on a grid_w-wide grid, then reference image
// tokens at (1, h, w) on a ref_w-wide grid.  Pair p belongs to axis 0 for
// p < a0/2, to axis 1 for p < (a0 + a1)/2, to axis 2 otherwise.
//
// A value depends only on (position along its axis, pair), so a CTA takes a
// kRopeTH x kRopeTW tile of one image grid, evaluates the distinct values of
// the tile once in fp64 (rows x axis-1 pairs, columns x axis-2 pairs, and
// the axis-0 pairs) into shared memory, and writes the tile's rows from
// there; text CTAs write the position-0 values (cos 1, sin 0) directly.
// FP64 is the slow unit of this GPU, and per-element evaluation cost about
// 13 times the evaluations.
constexpr int kRopeTH = 8, kRopeTW = 16, kRopeMaxAxisPairs = 64, kRopeTxtTok = 32;

__global__ void __launch_bounds__(256) rope_build_kernel(int L_txt, int grid_h, int grid_w, int ref_h, int ref_w,
                                                         int a0, int a1, int a2, double theta, int nb_txt,
                                                         int nt_gen_w, int nb_gen, int nt_ref_w,
                                                         int32_t* __restrict__ ids, float* __restrict__ cs,
                                                         float* __restrict__ sn) {
  __shared__ double om[3][kRopeMaxAxisPairs];
  __shared__ float tc[kRopeTH + kRopeTW + 1][kRopeMaxAxisPairs];
  __shared__ float ts[kRopeTH + kRopeTW + 1][kRopeMaxAxisPairs];
  const int npairs = (a0 + a1 + a2) / 2;
  const int e1 = a0 / 2, e2 = (a0 + a1) / 2;  // first pair of axis 1, of axis 2
  const int np0 = e1, np1 = e2 - e1, np2 = npairs - e2;
  int blk = (int)blockIdx.x;
  if (blk < nb_txt) {
    const long long tok0 = (long long)blk * kRopeTxtTok;
    for (int e = threadIdx.x; e < kRopeTxtTok * npairs; e += blockDim.x) {
      const long long tok = tok0 + e / npairs;
      const int p = e % npairs;
      if (tok >= L_txt) break;
      cs[tok * npairs + p] = 1.0f;  // cos(0), sin(0)
      sn[tok * npairs + p] = 0.0f;
      if (p == 0 && ids) ids[3 * tok] = 0, ids[3 * tok + 1] = 0, ids[3 * tok + 2] = 0;
    }
    return;
  }
  blk -= nb_txt;
  const int ref = blk >= nb_gen ? 1 : 0;
  if (ref) blk -= nb_gen;
  const int W = ref ? ref_w : grid_w, Hg = ref ? ref_h : grid_h, ntw = ref ? nt_ref_w : nt_gen_w;
  const long long base = (long long)L_txt + (ref ? (long long)grid_h * grid_w : 0);
  const int r0 = (blk / ntw) * kRopeTH, c0 = (blk % ntw) * kRopeTW;
  // frequencies of every pair, then the tile's distinct values
  for (int p = threadIdx.x; p < npairs; p += blockDim.x) {
    const int ax = p < e1 ? 0 : p < e2 ? 1 : 2;
    const int i = p - (ax == 0 ? 0 : ax == 1 ? e1 : e2);
    const int da = ax == 0 ? a0 : ax == 1 ? a1 : a2;
    om[ax][i] = pow(theta, (-2.0 * (double)i) / (double)da);
  }
  __syncthreads();
  const int n1 = kRopeTH * np1, n2 = kRopeTW * np2;
  for (int e = threadIdx.x; e < n1 + n2 + np0; e += blockDim.x) {
    int slot, i, ax, pos;
    if (e < n1) {
      slot = e / np1, i = e - slot * np1, ax = 1, pos = r0 + slot;
    } else if (e < n1 + n2) {
      const int f = e - n1, k = f / np2;
      slot = kRopeTH + k, i = f - k * np2, ax = 2, pos = c0 + k;
    } else {
      slot = kRopeTH + kRopeTW, i = e - n1 - n2, ax = 0, pos = ref;
    }
    const double ang = (double)pos * om[ax][i];
    tc[slot][i] = (float)cos(ang);
    ts[slot][i] = (float)sin(ang);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < kRopeTH * kRopeTW * npairs; e += blockDim.x) {
    const int t = e / npairs, p = e - t * npairs;
    const int r = r0 + t / kRopeTW, c = c0 + t % kRopeTW;
    if (r >= Hg || c >= W) continue;
    const long long tok = base + (long long)r * W + c;
    const int slot = p < e1 ? kRopeTH + kRopeTW : p < e2 ? r - r0 : kRopeTH + (c - c0);
    const int i = p < e1 ? p : p < e2 ? p - e1 : p - e2;
    cs[tok * npairs + p] = tc[slot][i];
    sn[tok * npairs + p] = ts[slot][i];
    if (p == 0 && ids) ids[3 * tok] = ref, ids[3 * tok + 1] = r, ids[3 * tok + 2] = c;
  }
}

// x [rows][row_stride] bf16, each row H*d channels; one thread per 8 channels.
__global__ void rope_apply_kernel(uint16_t* __restrict__ x, long long rows, int L, int H, int d, int row_stride,
                                  const float* __restrict__ cs, const float* __restrict__ sn) {
  const int chunks = H * d / 8;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * chunks) return;
  const long long row = idx / chunks;
  const int c = (int)(idx - row * chunks);
  const int tok = (int)(row % L);
  const int p0 = (c % (d / 8)) * 4;
  uint4* ptr = reinterpret_cast<uint4*>(x + row * row_stride + c * 8);
  uint4 v = *ptr;
  const float4 co = __ldg(reinterpret_cast<const float4*>(cs + (long long)tok * (d / 2) + p0));
  const float4 si = __ldg(reinterpret_cast<const float4*>(sn + (long long)tok * (d / 2) + p0));
  const float cc[4] = {co.x, co.y, co.z, co.w}, ss[4] = {si.x, si.y, si.z, si.w};
  uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float x0 = bf16_lo(u[j]), x1 = bf16_hi(u[j]);
    u[j] = pack_bf16x2(x0 * cc[j] - x1 * ss[j], x0 * ss[j] + x1 * cc[j]);
  }
  *ptr = make_uint4(u[0], u[1], u[2], u[3]);
}

// ------------------------------------------------------------------ Euler
// sig_tab != null: dt = sig_tab[k + 1] - sig_tab[k], k = *sig_idx, rounded once
// to fp32 (the same rounding as the host-side dt).
__device__ __forceinline__ float euler_dt(float dt, const double* sig_tab, const int* sig_idx) {
  if (!sig_tab) return dt;
  const int k = *sig_idx;
  return (float)(sig_tab[k + 1] - sig_tab[k]);
}

__global__ void euler_f32_kernel(float* __restrict__ x, const float* __restrict__ v, float dt,
                                 const double* __restrict__ sig_tab, const int* __restrict__ sig_idx, long long n) {
  dt = euler_dt(dt, sig_tab, sig_idx);
  const long long i = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i + 3 < n) {
    float4 a = *reinterpret_cast<float4*>(x + i);
    const float4 b = __ldg(reinterpret_cast<const float4*>(v + i));
    a.x = fmaf(dt, b.x, a.x), a.y = fmaf(dt, b.y, a.y), a.z = fmaf(dt, b.z, a.z), a.w = fmaf(dt, b.w, a.w);
    *reinterpret_cast<float4*>(x + i) = a;
  } else {
    for (long long k = i; k < n; ++k) x[k] = fmaf(dt, v[k], x[k]);
  }
}

__global__ void euler_bf16_kernel(float* __restrict__ x, const uint16_t* __restrict__ v, float dt,
                                  const double* __restrict__ sig_tab, const int* __restrict__ sig_idx, long long n) {
  dt = euler_dt(dt, sig_tab, sig_idx);
  const long long i = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i + 3 < n) {
    float4 a = *reinterpret_cast<float4*>(x + i);
    const uint2 b = __ldg(reinterpret_cast<const uint2*>(v + i));
    a.x = fmaf(dt, bf16_lo(b.x), a.x), a.y = fmaf(dt, bf16_hi(b.x), a.y);
    a.z = fmaf(dt, bf16_lo(b.y), a.z), a.w = fmaf(dt, bf16_hi(b.y), a.w);
    *reinterpret_cast<float4*>(x + i) = a;
  } else {
    for (long long k = i; k < n; ++k) x[k] = fmaf(dt, __uint_as_float((uint32_t)v[k] << 16), x[k]);
  }
}

// ------------------------------------------------------------------ int8
template <typename T>
__device__ __forceinline__ float load_w(const T* w, long long i);
template <>
__device__ __forceinline__ float load_w<float>(const float* w, long long i) {
  return w[i];
}
template <>
__device__ __forceinline__ float load_w<uint16_t>(const uint16_t* w, long long i) {
  return __uint_as_float((uint32_t)w[i] << 16);
}

// One CTA per output row: s = max|w| / 127 (fp32), q = clamp(rint(w / s)).
template <typename T>
__global__ void __launch_bounds__(256) quantize_kernel(const T* __restrict__ w, int K, int8_t* __restrict__ q,
                                                       float* __restrict__ scale) {
  __shared__ float red[8];
  const long long base = (long long)blockIdx.x * K;
  float m = 0.f;
  for (int k = threadIdx.x; k < K; k += blockDim.x) m = fmaxf(m, fabsf(load_w<T>(w, base + k)));
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    t = warp_max(t);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  const float amax = red[0];
  const float s = amax == 0.f ? 1.0f : __fdiv_rn(amax, 127.0f);
  if (threadIdx.x == 0) scale[blockIdx.x] = s;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    float r = rintf(__fdiv_rn(load_w<T>(w, base + k), s));
    r = fminf(fmaxf(r, -127.f), 127.f);
    q[base + k] = (int8_t)r;
  }
}

// One CTA per row of x (row stride ld): s = max|x| / 448 (fp32, 1 for a zero
// row), q = e4m3(x / s) with the quotient rounded once in fp32.  K even.
template <typename T>
__global__ void __launch_bounds__(256) quantize_f8_kernel(const T* __restrict__ x, long long ld, int K,
                                                          uint8_t* __restrict__ q, long long qld,
                                                          float* __restrict__ scale) {
  __shared__ float red[8];
  const T* row = x + (long long)blockIdx.x * ld;
  uint8_t* qrow = q + (long long)blockIdx.x * qld;
  float m = 0.f;
  for (int k = threadIdx.x; k < K; k += blockDim.x) m = fmaxf(m, fabsf(load_w<T>(row, k)));
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    t = warp_max(t);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  const float amax = red[0];
  const float s = amax == 0.f ? 1.0f : __fdiv_rn(amax, 448.0f);
  if (threadIdx.x == 0) scale[blockIdx.x] = s;
  for (int k = 2 * threadIdx.x; k < K; k += 2 * blockDim.x)
    *reinterpret_cast<uint16_t*>(qrow + k) =
        f8x2_e4m3(__fdiv_rn(load_w<T>(row, k), s), __fdiv_rn(load_w<T>(row, k + 1), s));
}

// The same for bf16 rows read once: each thread holds CPT 16-byte chunks (8
// values) of the row in registers, so the row is read from memory once and
// written once as e4m3.  K a multiple of 8, K <= 2048 CPT; row starts 16-byte
// aligned.
template <int CPT>
__global__ void __launch_bounds__(256) quantize_f8_bf16_kernel(const uint16_t* __restrict__ x, long long ld, int K,
                                                               uint8_t* __restrict__ q, long long qld,
                                                               float* __restrict__ scale) {
  __shared__ float red[8];
  const int nch = K / 8;
  const uint4* row = reinterpret_cast<const uint4*>(x + (long long)blockIdx.x * ld);
  uint2* qrow = reinterpret_cast<uint2*>(q + (long long)blockIdx.x * qld);
  uint4 v[CPT];
  float m = 0.f;
#pragma unroll
  for (int c = 0; c < CPT; ++c) {
    const int i = threadIdx.x + c * 256;
    v[c] = i < nch ? __ldg(row + i) : make_uint4(0, 0, 0, 0);
    const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
  }
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < 8 ? red[threadIdx.x] : 0.f;
    t = warp_max(t);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  const float amax = red[0];
  const float s = amax == 0.f ? 1.0f : __fdiv_rn(amax, 448.0f);
  if (threadIdx.x == 0) scale[blockIdx.x] = s;
#pragma unroll
  for (int c = 0; c < CPT; ++c) {
    const int i = threadIdx.x + c * 256;
    if (i < nch) {
      const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
      uint16_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) o[j] = f8x2_e4m3(__fdiv_rn(bf16_lo(w[j]), s), __fdiv_rn(bf16_hi(w[j]), s));
      qrow[i] = make_uint2((uint32_t)o[0] | ((uint32_t)o[1] << 16), (uint32_t)o[2] | ((uint32_t)o[3] << 16));
    }
  }
}

// int8 -> bf16 (exact: |q| <= 127 has at most 7 significant bits); 16 per thread.
__global__ void dequant_i8_kernel(const int8_t* __restrict__ q, uint16_t* __restrict__ out, long long n16) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n16) return;
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(q) + i);
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float lo = (float)(int8_t)((u[j >> 1] >> (16 * (j & 1))) & 0xFF);
    const float hi = (float)(int8_t)((u[j >> 1] >> (16 * (j & 1) + 8)) & 0xFF);
    o[j] = pack_bf16x2(lo, hi);
  }
  uint4* d = reinterpret_cast<uint4*>(out) + 2 * i;
  d[0] = make_uint4(o[0], o[1], o[2], o[3]);
  d[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

__global__ void cast_f32_bf16_kernel(const float* __restrict__ x, uint16_t* __restrict__ y, long long n4) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const float4 v = __ldg(reinterpret_cast<const float4*>(x) + i);
  reinterpret_cast<uint2*>(y)[i] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
}

// ------------------------------------------------------------------ attention prep
// One warp per (sample, token, head): q and k get RMSNorm (gain by stream)
// and RoPE, written to qk [B][L][2D].  v goes transposed to vT [B][D][Lpad]
// through vT_transpose_kernel below.
template <int HD>
__global__ void attn_prep_kernel(const uint16_t* __restrict__ qkv, long long qkv_ld, int B, int L, int L_txt, int H,
                                 const float* gq0, const float* gq1, const float* gk0, const float* gk1, float eps,
                                 const float* __restrict__ cs, const float* __restrict__ sn, uint16_t* __restrict__ qk) {
  constexpr int PER = HD / 32;  // channels per lane (2 or 4), consecutive
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= (long long)B * L * H) return;
  const int h = (int)(gw % H);
  const long long bt = gw / H;
  const int tok = (int)(bt % L);
  const int D = H * HD;
  const uint16_t* row = qkv + bt * qkv_ld;
  const bool txt = tok < L_txt;
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const float* g = which == 0 ? (txt ? gq0 : gq1) : (txt ? gk0 : gk1);
    const uint16_t* src = row + which * D + h * HD + lane * PER;
    float v[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) v[j] = __uint_as_float((uint32_t)src[j] << 16);
    if (g) {
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < PER; ++j) ss = fmaf(v[j], v[j], ss);
      const float rs = rsqrtf(warp_sum(ss) * (1.0f / HD) + eps);
#pragma unroll
      for (int j = 0; j < PER; ++j) v[j] = v[j] * rs * g[lane * PER + j];
    }
    if (cs) {
#pragma unroll
      for (int j = 0; j < PER; j += 2) {
        const int pr = (lane * PER + j) / 2;
        const float c = cs[(long long)tok * (HD / 2) + pr], s = sn[(long long)tok * (HD / 2) + pr];
        const float x0 = v[j], x1 = v[j + 1];
        v[j] = x0 * c - x1 * s;
        v[j + 1] = x0 * s + x1 * c;
      }
    }
    uint16_t* dst = qk + bt * (2LL * D) + which * D + h * HD + lane * PER;
#pragma unroll
    for (int j = 0; j < PER; j += 2) *reinterpret_cast<uint32_t*>(dst + j) = pack_bf16x2(v[j], v[j + 1]);
  }
}

// V^T for the standalone attention: v[b][tok][c] (columns 2D + c of a qkv
// row) -> vT[b][c][tok].  A CTA moves a 64-token x 64-channel tile through
// shared memory, so that the loads (8 channels of one token) and the stores
// (8 tokens of one channel) are 16-byte vectors along contiguous memory.
// In the tile, the 16-byte chunk j of token row r sits at chunk position
// j ^ ((r >> 3) & 7): the 8-token chunks one warp reads for a channel are
// 8 rows apart, and the swizzle puts them in 8 different bank groups.
// Tokens at or beyond L load as zeros and are stored only up to the 8-token
// chunk holding token L - 1 (vT rows are padded to a multiple of 8).
__global__ void __launch_bounds__(256) vT_transpose_kernel(const uint16_t* __restrict__ qkv, long long qkv_ld, int L,
                                                           int D, uint16_t* __restrict__ vT, long long vT_ld) {
  __shared__ __align__(16) uint16_t tile[64][64];  // [token][channel], swizzled 16-byte chunks
  const int t0 = blockIdx.x * 64, c0 = blockIdx.y * 64, b = blockIdx.z;
  for (int i = threadIdx.x; i < 64 * 8; i += 256) {
    const int t = i >> 3, k = i & 7;  // token of the tile, 8-channel chunk
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (t0 + t < L)
      v = *reinterpret_cast<const uint4*>(qkv + ((long long)b * L + t0 + t) * qkv_ld + 2LL * D + c0 + 8 * k);
    *reinterpret_cast<uint4*>(&tile[t][8 * (k ^ ((t >> 3) & 7))]) = v;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 64 * 8; i += 256) {
    const int c = i >> 3, t = 8 * (i & 7);  // channel of the tile, first token of an 8-token chunk
    if (t0 + t >= L) continue;
    const int col = 8 * ((c >> 3) ^ ((t >> 3) & 7)) + (c & 7);  // rows t .. t + 7 share t >> 3
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = (uint32_t)tile[t + 2 * q][col] | ((uint32_t)tile[t + 2 * q + 1][col] << 16);
    *reinterpret_cast<uint4*>(vT + ((long long)b * D + c0 + c) * vT_ld + t0 + t) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ------------------------------------------------------------------ wait self-test
// Waits on an mbarrier that nothing ever completes, with the given limit:
// exercises the bounded-wait path (status bit, abort flag, orderly exit).
__global__ void wait_selftest_kernel(unsigned long long limit_ns, unsigned* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  mbar_wait(smem_u32(&bar), 0, &abort_flag, status, ST_SELFTEST, limit_ns);
  __syncthreads();
}

}  // namespace

// ------------------------------------------------------------------ launchers
cudaError_t launch_wait_selftest(unsigned long long limit_ns, unsigned* status, cudaStream_t st) {
  launch_begin(KID_SELFTEST, st);
  wait_selftest_kernel<<<1, 32, 0, st>>>(limit_ns, status);
  launch_end(st);
  return cudaGetLastError();
}

cudaError_t launch_ln_modulate_jobs(const LnJob* jobs, int n_jobs, int D, float eps, cudaStream_t st) {
  // D / 128 is then one of the even cases 2 .. 32 below
  if (D % 256 || D < 256 || D > 4096 || n_jobs < 1 || n_jobs > 2) return cudaErrorInvalidValue;
  LnJobs J;
  J.n0 = 0;
  J.n_total = 0;
  J.eps = eps;
  bool f8 = false;
  for (int k = 0; k < n_jobs; ++k) {
    const LnJob& jo = jobs[k];
    if (jo.rows < 1 || jo.n_seg < 1) return cudaErrorInvalidValue;
    if ((jo.q == nullptr) != (jo.qs == nullptr) || (!jo.q && !jo.y)) return cudaErrorInvalidValue;
    if (k > 0 && (jo.q != nullptr) != f8) return cudaErrorInvalidValue;  // one output kind per launch
    f8 = jo.q != nullptr;
    J.job[k] = jo;
    J.n_total += jo.rows * jo.n_seg;
    if (k == 0) J.n0 = J.n_total;
  }
  if (n_jobs == 1) J.job[1] = J.job[0];
  const int blocks = (J.n_total + 3) / 4;  // four rows (warps) per CTA
  launch_begin(KID_LN_MODULATE, st);
  switch (D / 128) {
#define MMDIT_LN_CASE(nv)                                        \
  case nv:                                                       \
    if (f8)                                                      \
      ln_mod_kernel<nv, true><<<blocks, 128, 0, st>>>(J);        \
    else                                                         \
      ln_mod_kernel<nv, false><<<blocks, 128, 0, st>>>(J);       \
    break;
    MMDIT_LN_CASE(2) MMDIT_LN_CASE(4) MMDIT_LN_CASE(6) MMDIT_LN_CASE(8) MMDIT_LN_CASE(10) MMDIT_LN_CASE(12)
    MMDIT_LN_CASE(14) MMDIT_LN_CASE(16) MMDIT_LN_CASE(18) MMDIT_LN_CASE(20) MMDIT_LN_CASE(22) MMDIT_LN_CASE(24)
    MMDIT_LN_CASE(26) MMDIT_LN_CASE(28) MMDIT_LN_CASE(30) MMDIT_LN_CASE(32)
#undef MMDIT_LN_CASE
    default:
      break;
  }
  launch_end(st);
  return cudaGetLastError();
}

cudaError_t launch_ln_modulate(const float* x, long long x_seg_rows, int rows, int n_seg, int D, const float* shift,
                               const float* scale, long long mod_stride, float eps, uint16_t* y, cudaStream_t st,
                               uint8_t* q, float* qs) {
  LnJob jo{x, x_seg_rows, rows, n_seg, shift, scale, mod_stride, y, q, qs};
  return launch_ln_modulate_jobs(&jo, 1, D, eps, st);
}

// CTAs of a GEMV kernel that are resident at once (the grid-stride loop
// wants no second wave).  Cached per (kernel, shared memory), so launches
// inside a stream capture make no query.
static int gemv_resident_ctas(const void* kern, size_t smem) {
  static std::mutex mu;
  static struct {
    const void* k;
    size_t smem;
    int dev, n;
  } cache[32];
  static int n_cache = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_cache; ++i)
    if (cache[i].k == kern && cache[i].smem == smem && cache[i].dev == dev) return cache[i].n;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, smem) != cudaSuccess || per_sm < 1) {
    (void)cudaGetLastError();
    per_sm = 1;
  }
  if (per_sm > kGemvCtasPerSm) per_sm = kGemvCtasPerSm;
  const int n = per_sm * num_sms();
  if (n_cache < 32) cache[n_cache++] = {kern, smem, dev, n};
  return n;
}

// The kernel instance for B rows of x: the smallest batch bound >= B.
using GemvFn = void (*)(const void*, const float*, const float*, const float*, int, int, int, int, float*);
using GemvBatchedFn = void (*)(const GemvBatch, const float*, int, int, int);
template <bool I8>
static GemvFn gemv_fn(int B) {
  return B <= 1   ? gemv_kernel<I8, 1>
         : B <= 2 ? gemv_rows_kernel<I8, 2>
         : B <= 4 ? gemv_rows_kernel<I8, 4>
                  : gemv_rows_kernel<I8, 8>;
}
template <bool I8>
static GemvBatchedFn gemv_batched_fn(int B) {
  return B <= 1   ? gemv_batched_kernel<I8, 1>
         : B <= 2 ? gemv_rows_batched_kernel<I8, 2>
         : B <= 4 ? gemv_rows_batched_kernel<I8, 4>
                  : gemv_rows_batched_kernel<I8, 8>;
}

// Lets every GEMV instance use up to 200 KB of dynamic shared memory (x of up
// to 8 rows); once per device, safe under concurrent first calls.
static cudaError_t gemv_attributes() {
  static std::once_flag once[64];
  static cudaError_t err[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::call_once(once[dev], [&] {
    err[dev] = cudaSuccess;
    for (int B : {1, 2, 4, 8}) {
      const void* fns[4] = {(const void*)gemv_fn<false>(B), (const void*)gemv_fn<true>(B),
                            (const void*)gemv_batched_fn<false>(B), (const void*)gemv_batched_fn<true>(B)};
      for (const void* f : fns) {
        const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e != cudaSuccess && err[dev] == cudaSuccess) err[dev] = e;
      }
    }
  });
  return err[dev];
}

static cudaError_t launch_gemv_batched_rows(const GemvJob* jobs, int n_jobs, bool i8, const float* x, int r0, int B,
                                           int K, int act, cudaStream_t st);

// The kernels take at most kGemvMaxRows rows of x (their compile-time batch
// bound); more rows go in consecutive launches of up to that many.
constexpr int kGemvMaxRows = 8;

cudaError_t launch_gemv(const void* W, bool i8, const float* wscale, const float* bias, const float* x, int B, int N,
                        int K, int act, float* y, cudaStream_t st) {
  const cudaError_t ea = gemv_attributes();
  if (ea != cudaSuccess) return ea;
  for (int r0 = 0; r0 < B; r0 += kGemvMaxRows) {
    const int nb = B - r0 < kGemvMaxRows ? B - r0 : kGemvMaxRows;
    const size_t smem = (size_t)nb * K * sizeof(float);
    const GemvFn fn = i8 ? gemv_fn<true>(nb) : gemv_fn<false>(nb);
    const int rows_per_cta = kGemvWarps * kGemvRowsPerWarp;
    int blocks = (N + rows_per_cta - 1) / rows_per_cta;
    const int resident = gemv_resident_ctas((const void*)fn, smem);
    if (blocks > resident) blocks = resident;
    launch_begin(KID_GEMV, st);
    fn<<<blocks, 256, smem, st>>>(W, wscale, bias, x + (size_t)r0 * K, nb, N, K, act, y + (size_t)r0 * N);
    launch_end(st);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_gemv_batched(const GemvJob* jobs, int n_jobs, bool i8, const float* x, int B, int K, int act,
                                cudaStream_t st) {
  const cudaError_t ea = gemv_attributes();
  if (ea != cudaSuccess) return ea;
  for (int r0 = 0; r0 < B; r0 += kGemvMaxRows) {
    const int nb = B - r0 < kGemvMaxRows ? B - r0 : kGemvMaxRows;
    const cudaError_t e = launch_gemv_batched_rows(jobs, n_jobs, i8, x + (size_t)r0 * K, r0, nb, K, act, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Rows r0 .. r0 + B - 1 of x (x points at row r0), B <= kGemvMaxRows.
static cudaError_t launch_gemv_batched_rows(const GemvJob* jobs, int n_jobs, bool i8, const float* x, int r0, int B,
                                           int K, int act, cudaStream_t st) {
  const size_t smem = (size_t)B * K * sizeof(float);
  const GemvBatchedFn fn = i8 ? gemv_batched_fn<true>(B) : gemv_batched_fn<false>(B);
  for (int first = 0; first < n_jobs; first += kMaxGemvJobs) {
    GemvBatch jb;
    jb.n_jobs = n_jobs - first < kMaxGemvJobs ? n_jobs - first : kMaxGemvJobs;
    jb.row0[0] = 0;
    for (int i = 0; i < jb.n_jobs; ++i) {
      jb.job[i] = jobs[first + i];
      const long long ldo = jb.job[i].ldo ? jb.job[i].ldo : jb.job[i].N;
      jb.job[i].out += (size_t)r0 * ldo;
      jb.row0[i + 1] = jb.row0[i] + jobs[first + i].N;
    }
    for (int i = jb.n_jobs; i < kMaxGemvJobs; ++i) {
      jb.job[i] = GemvJob{nullptr, nullptr, nullptr, nullptr, 0, 0};
      jb.row0[i + 1] = jb.row0[jb.n_jobs];
    }
    const int rows_per_cta = kGemvWarps * kGemvRowsPerWarp;
    int blocks = (jb.row0[jb.n_jobs] + rows_per_cta - 1) / rows_per_cta;
    const int resident = gemv_resident_ctas((const void*)fn, smem);
    if (blocks > resident) blocks = resident;
    launch_begin(KID_GEMV, st);
    fn<<<blocks, 256, smem, st>>>(jb, x, B, K, act);
    launch_end(st);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_sinusoid(double t, int B, int dim, float* out, cudaStream_t st, const double* t_tab,
                            const int* t_idx, double t_scale) {
  const int n = B * dim;
  launch_begin(KID_SINUSOID, st);
  sinusoid_kernel<<<(n + 255) / 256, 256, 0, st>>>(t, t_tab, t_idx, t_scale, B, dim, out);
  launch_end(st);
  return cudaGetLastError();
}

cudaError_t launch_rope_build(int L_txt, int grid_w, int n_gen, int ref_w, int L, const int axes[3], double theta,
                              int32_t* ids, float* cs,
                              float* sn, cudaStream_t st) {
  const int npairs = (axes[0] + axes[1] + axes[2]) / 2;
  if (axes[0] / 2 > kRopeMaxAxisPairs || (axes[0] + axes[1]) / 2 - axes[0] / 2 > kRopeMaxAxisPairs ||
      npairs - (axes[0] + axes[1]) / 2 > kRopeMaxAxisPairs || grid_w < 1)
    return cudaErrorInvalidValue;
  const int grid_h = n_gen / grid_w;
  const int n_ref = L - L_txt - n_gen;
  const int rw = ref_w > 0 ? ref_w : 1, rh = n_ref > 0 ? n_ref / rw : 0;
  const int nb_txt = (L_txt + kRopeTxtTok - 1) / kRopeTxtTok;
  const int nt_gen_w = (grid_w + kRopeTW - 1) / kRopeTW, nt_ref_w = (rw + kRopeTW - 1) / kRopeTW;
  const int nb_gen = ((grid_h + kRopeTH - 1) / kRopeTH) * nt_gen_w;
  const int nb_ref = rh > 0 ? ((rh + kRopeTH - 1) / kRopeTH) * nt_ref_w : 0;
  const int blocks = nb_txt + nb_gen + nb_ref;
  if (blocks == 0) return cudaSuccess;
  launch_begin(KID_ROPE_BUILD, st);
  rope_build_kernel<<<blocks, 256, 0, st>>>(L_txt, grid_h, grid_w, rh, rw, axes[0], axes[1], axes[2], theta, nb_txt,
                                            nt_gen_w, nb_gen, nt_ref_w, ids, cs, sn);
  launch_end(st);
  return cudaGetLastError();
}

cudaError_t launch_heads_pack(const uint16_t* src, long long rows, int src_ld, int sections, int groups, int gc,
                              uint16_t* dst, cudaStream_t st) {
  const long long n = rows * sections * groups * (gc / 8);
  if (n == 0) return cudaSuccess;
  launch_begin(KID_HEADS_PACK, st);
  const unsigned grid = (unsigned)std::min<long long>(rows, (long long)num_sms() * 8);
  heads_pack_kernel<<<grid, 256, 0, st>>>(src, rows, src_ld, sections, groups, gc, dst);
  launch_end(st);
  return cudaGetLastError();
}

cudaError_t launch_heads_unpack(const uint16_t* src, long long rows, int groups, int gc, uint16_t* dst, int dst_ld,
                                cudaStream_t st) {
  const long long n = rows * groups * (gc / 8);
  if (n == 0) return cudaSuccess;
  launch_begin(KID_HEADS_UNPACK, st);
  const unsigned grid = (unsigned)std::min<long long>(rows, (long long)num_sms() * 8);
  heads_unpack_kernel<<<grid, 256, 0, st>>>(src, rows, groups, gc, dst, dst_ld);
  launch_end(st);
  return cudaGetLastError();
}

cudaError_t launch_rope_apply(uint16_t* x, long long rows, int L, int H, int d, int row_stride, const float* cs,
                              const float* sn, cudaStream_t st) {
  const long long n = rows * (H * d / 8);
  launch_begin(KID_ROPE_APPLY, st);
  rope_apply_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(x, rows, L, H, d, row_stride, cs, sn);
  launch_end(st);
  return cudaGetLastError();
}

cudaError_t launch_euler(float* x, const void* v, bool v_bf16, float dt, long long n, cudaStream_t st,
                         const double* sig_tab, const int* sig_idx) {
  const long long threads = (n + 3) / 4;
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  launch_begin(KID_EULER, st);
  if (v_bf16)
    euler_bf16_kernel<<<blocks, 256, 0, st>>>(x, reinterpret_cast<const uint16_t*>(v), dt, sig_tab, sig_idx, n);
  else
    euler_f32_kernel<<<blocks, 256, 0, st>>>(x, reinterpret_cast<const float*>(v), dt, sig_tab, sig_idx, n);
  launch_end(st);
  return cudaGetLastError();
}

cudaError_t launch_add(float* y, const float* x, long long n, cudaStream_t st) {
  launch_begin(KID_ADD, st);
  add_f32_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(y, x, n);
  launch_end(st);
  return cudaGetLastError();
}

cudaError_t launch_select_step(const float* src, long long stride, long long n, const int* k_dev, int k_host,
                               float* dst, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  if (n % 4 || stride % 4 || (reinterpret_cast<uintptr_t>(src) & 15) || (reinterpret_cast<uintptr_t>(dst) & 15))
    return cudaErrorInvalidValue;
  const long long n4 = n / 4;
  long long blocks = (n4 + 255) / 256;
  if (blocks > 4 * num_sms()) blocks = 4 * num_sms();
  launch_begin(KID_SELECT_STEP, st);
  select_step_kernel<<<(unsigned)blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(src), stride / 4, n4, k_dev,
                                                        k_host, reinterpret_cast<float4*>(dst));
  launch_end(st);
  return cudaGetLastError();
}

cudaError_t launch_counter(int* c, int value, bool add, cudaStream_t st) {
  launch_begin(KID_COUNTER, st);
  counter_kernel<<<1, 1, 0, st>>>(c, value, add ? 1 : 0);
  launch_end(st);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const void* w, bool w_bf16, int N, int K, int8_t* q, float* scale, cudaStream_t st) {
  launch_begin(KID_QUANTIZE, st);
  if (w_bf16)
    quantize_kernel<uint16_t><<<N, 256, 0, st>>>(reinterpret_cast<const uint16_t*>(w), K, q, scale);
  else
    quantize_kernel<float><<<N, 256, 0, st>>>(reinterpret_cast<const float*>(w), K, q, scale);
  launch_end(st);
  return cudaGetLastError();
}

cudaError_t launch_quantize_f8(const void* x, bool x_bf16, long long rows, int K, long long ld, uint8_t* q,
                               long long qld, float* scale, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  launch_begin(KID_QUANTIZE_F8, st);
  const bool vec = x_bf16 && K % 8 == 0 && K <= 2048 * 8 && ld % 8 == 0 && qld % 8 == 0 &&
                   (reinterpret_cast<uintptr_t>(x) & 15) == 0 && (reinterpret_cast<uintptr_t>(q) & 7) == 0;
  if (vec) {
    const uint16_t* xb = reinterpret_cast<const uint16_t*>(x);
    const int cpt = (K / 8 + 255) / 256;
    if (cpt <= 1)
      quantize_f8_bf16_kernel<1><<<(unsigned)rows, 256, 0, st>>>(xb, ld, K, q, qld, scale);
    else if (cpt <= 2)
      quantize_f8_bf16_kernel<2><<<(unsigned)rows, 256, 0, st>>>(xb, ld, K, q, qld, scale);
    else if (cpt <= 4)
      quantize_f8_bf16_kernel<4><<<(unsigned)rows, 256, 0, st>>>(xb, ld, K, q, qld, scale);
    else
      quantize_f8_bf16_kernel<8><<<(unsigned)rows, 256, 0, st>>>(xb, ld, K, q, qld, scale);
  } else if (x_bf16)
    quantize_f8_kernel<uint16_t><<<(unsigned)rows, 256, 0, st>>>(reinterpret_cast<const uint16_t*>(x), ld, K, q, qld,
                                                                  scale);
  else
    quantize_f8_kernel<float><<<(unsigned)rows, 256, 0, st>>>(reinterpret_cast<const float*>(x), ld, K, q, qld, scale);
  launch_end(st);
  return cudaGetLastError();
}

cudaError_t launch_dequant_i8(const int8_t* q, uint16_t* out, long long n, cudaStream_t st) {
  const long long n16 = n / 16;
  launch_begin(KID_DEQUANT, st);
  dequant_i8_kernel<<<(unsigned)((n16 + 255) / 256), 256, 0, st>>>(q, out, n16);
  launch_end(st);
  return cudaGetLastError();
}

cudaError_t launch_cast_bf16(const float* x, uint16_t* y, long long n, cudaStream_t st) {
  const long long n4 = n / 4;
  launch_begin(KID_CAST, st);
  cast_f32_bf16_kernel<<<(unsigned)((n4 + 255) / 256), 256, 0, st>>>(x, y, n4);
  launch_end(st);
  return cudaGetLastError();
}

cudaError_t launch_attn_prep(const uint16_t* qkv, long long qkv_ld, int B, int L, int L_txt, int H, int d,
                             const float* gq0, const float* gq1, const float* gk0, const float* gk1, float eps,
                             const float* cs, const float* sn, uint16_t* qk, uint16_t* vT, long long vT_ld,
                             cudaStream_t st) {
  const long long warps = (long long)B * L * H;
  const unsigned blocks = (unsigned)((warps * 32 + 255) / 256);
  launch_begin(KID_ATTN_PREP, st);
  if (d == 128)
    attn_prep_kernel<128><<<blocks, 256, 0, st>>>(qkv, qkv_ld, B, L, L_txt, H, gq0, gq1, gk0, gk1, eps, cs, sn, qk);
  else
    attn_prep_kernel<64><<<blocks, 256, 0, st>>>(qkv, qkv_ld, B, L, L_txt, H, gq0, gq1, gk0, gk1, eps, cs, sn, qk);
  launch_end(st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int D = H * d;
  launch_begin(KID_VT_TRANSPOSE, st);
  vT_transpose_kernel<<<dim3((unsigned)((L + 63) / 64), (unsigned)(D / 64), (unsigned)B), 256, 0, st>>>(qkv, qkv_ld, L,
                                                                                                    D, vT, vT_ld);
  launch_end(st);
  return cudaGetLastError();
}

}  // namespace mmdit
