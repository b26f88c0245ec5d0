// Flash-style joint softmax attention on tcgen05 (sm_103a).
//
// Computes softmax(q k^T / sqrt(d)) v per (sample, head) over the whole
// concatenated [text; image] sequence with no mask: the scores, scale, max,
// exponent, sum and divide of the attention definition in the Luminal blog
// (section "What the compiler found on its own"), evaluated tile by tile
// with an online (running max / running sum) softmax so that the L x L score
// matrix never leaves the SM.
//
// Inputs are already RMS-normalised and rotated (the producing GEMM's
// epilogue, or the prep kernel of joint_attention_fwd, does that once per
// token instead of once per query tile): q and k rows in a [B][L][2D] buffer
// (q at column h*d, k at column D + h*d), v transposed as [B][D][Lpad] so
// that both MMAs read K-major operands.
//
// CTA = 128 queries of one (sample, head); 192 threads:
//   warp 0      TMA: Q once, then K and V^T tiles of 128 keys, 2-stage ring.
//   warp 1      TMEM (512 columns: S double buffer 2x128, O d columns) and
//               the MMAs S = Q K^T (M=128, N=128, K=d) and O += P V
//               (M=128, N=d, K=128) from one thread.
//   warps 2-5   softmax, one query row per thread: tcgen05.ld of the S row,
//               running max in the log2 domain, exp2 on the MUFU, P written
//               to shared memory in the swizzled K-major layout, O rescaled
//               in TMEM only when the running max grows by more than 2^8,
//               final O / l and bf16 store.
#include "common.cuh"

namespace mmdit {

namespace {

constexpr int kAttnThreads = 192;
constexpr uint32_t kHalf = 128 * 128;  // one 128-row x 128-byte swizzled half tile
constexpr float kRescaleThreshold = 8.0f;

template <int HD>
struct AttnSmem {
  static constexpr uint32_t Q = (HD / 64) * kHalf;
  static constexpr uint32_t K = (HD / 64) * kHalf;
  static constexpr uint32_t V = 2 * HD * 128;  // two 64-key halves of HD rows x 128 B
  static constexpr uint32_t P = 2 * kHalf;
  static constexpr uint32_t total = 1024 + Q + 2 * K + 2 * V + P + 256;
};

template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ AttnParams p) {
  using SM = AttnSmem<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + SM::Q;
  uint8_t* sV = sK + 2 * SM::K;
  uint8_t* sP = sV + 2 * SM::V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + SM::P);
  const uint32_t q_full = smem_u32(bars + 0);
  const uint32_t k_full0 = smem_u32(bars + 1);   // [2]
  const uint32_t v_full0 = smem_u32(bars + 3);   // [2]
  const uint32_t kv_empty0 = smem_u32(bars + 5); // [2]
  const uint32_t s_full0 = smem_u32(bars + 7);   // [2]
  const uint32_t s_empty0 = smem_u32(bars + 9);  // [2]
  const uint32_t p_full = smem_u32(bars + 11);
  const uint32_t pv_done = smem_u32(bars + 12);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 13);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int q0 = qt * kAttnBM;
  const int D = p.H * HD;
  const int nkv = p.n_kv_tiles;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(k_full0 + 8 * i, 1);
      mbar_init(v_full0 + 8 * i, 1);
      mbar_init(kv_empty0 + 8 * i, 1);
      mbar_init(s_full0 + 8 * i, 1);
      mbar_init(s_empty0 + 8 * i, 4);
    }
    mbar_init(p_full, 4);
    mbar_init(pv_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_O = tmem + 256;

  if (warp == 0) {
    if (lane == 0) {
      mbar_expect_tx(q_full, SM::Q);
#pragma unroll
      for (int hf = 0; hf < HD / 64; ++hf)
        tma_load_3d(smem_u32(sQ + hf * kHalf), &tmQK, q_full, h * HD + hf * 64, q0, b);
      for (int j = 0; j < nkv; ++j) {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!mbar_wait(kv_empty0 + 8 * st, ph ^ 1, abort_flag, p.status, ST_TIMEOUT_PRODUCER)) break;
        mbar_expect_tx(k_full0 + 8 * st, SM::K);
#pragma unroll
        for (int hf = 0; hf < HD / 64; ++hf)
          tma_load_3d(smem_u32(sK + st * SM::K + hf * kHalf), &tmQK, k_full0 + 8 * st, D + h * HD + hf * 64,
                      j * kAttnBN, b);
        mbar_expect_tx(v_full0 + 8 * st, SM::V);
#pragma unroll
        for (int kh = 0; kh < 2; ++kh)
          tma_load_3d(smem_u32(sV + st * SM::V + kh * (HD * 128)), &tmV, v_full0 + 8 * st, j * kAttnBN + kh * 64,
                      h * HD, b);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16(128, kAttnBN);
      const uint32_t idesc_o = idesc_bf16(128, HD);
      bool ok = mbar_wait(q_full, 0, abort_flag, p.status, ST_TIMEOUT_MMA);
      const uint32_t aQ = smem_u32(sQ);
      auto issue_pv = [&](int i) -> bool {
        const int st = i & 1;
        if (!mbar_wait(p_full, i & 1, abort_flag, p.status, ST_TIMEOUT_MMA)) return false;
        if (!mbar_wait(v_full0 + 8 * st, (i >> 1) & 1, abort_flag, p.status, ST_TIMEOUT_MMA)) return false;
        tc_fence_after();
        const uint32_t aP = smem_u32(sP);
        const uint32_t bV = smem_u32(sV + st * SM::V);
#pragma unroll
        for (int k = 0; k < kAttnBN / 16; ++k) {
          const int kh = k >> 2, off = (k & 3) * 32;
          umma_bf16(tmem_O, sdesc_k128(aP + kh * kHalf + off), sdesc_k128(bV + kh * (HD * 128) + off), idesc_o,
                    (i > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(pv_done);
        umma_commit(kv_empty0 + 8 * st);
        return true;
      };
      for (int j = 0; ok && j < nkv; ++j) {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!mbar_wait(k_full0 + 8 * st, ph, abort_flag, p.status, ST_TIMEOUT_MMA)) { ok = false; break; }
        if (!mbar_wait(s_empty0 + 8 * st, ph ^ 1, abort_flag, p.status, ST_TIMEOUT_MMA)) { ok = false; break; }
        tc_fence_after();
        const uint32_t bK = smem_u32(sK + st * SM::K);
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const int hf = k >> 2, off = (k & 3) * 32;
          umma_bf16(tmem + st * kAttnBN, sdesc_k128(aQ + hf * kHalf + off), sdesc_k128(bK + hf * kHalf + off),
                    idesc_s, k > 0 ? 1u : 0u);
        }
        umma_commit(s_full0 + 8 * st);
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok) issue_pv(nkv - 1);
    }
  } else {
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    float m_run = -INFINITY, l_run = 0.f;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int st = j & 1;
      if (!mbar_wait(s_full0 + 8 * st, (j >> 1) & 1, abort_flag, p.status, ST_TIMEOUT_SOFTMAX)) { ok = false; break; }
      tc_fence_after();
      float s[kAttnBN];
#pragma unroll
      for (int c = 0; c < kAttnBN / 32; ++c) {
        uint32_t raw[32];
        MMDIT_TMEM_LD32(tmem + lane_base + st * kAttnBN + c * 32, raw);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(raw[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty0 + 8 * st);
      const int kv0 = j * kAttnBN;
      if (kv0 + kAttnBN > p.L) {
#pragma unroll
        for (int c = 0; c < kAttnBN; ++c)
          if (kv0 + c >= p.L) s[c] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < kAttnBN; ++c) mx = fmaxf(mx, s[c]);
      const float m_new = fmaxf(m_run, mx * sl2);
      if (j > 0) {
        if (!mbar_wait(pv_done, (j - 1) & 1, abort_flag, p.status, ST_TIMEOUT_SOFTMAX)) { ok = false; break; }
        tc_fence_after();
      }
      if (m_new > m_run + kRescaleThreshold) {
        const float alpha = ex2_approx(m_run - m_new);
        if (j > 0) {
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t raw[32];
            MMDIT_TMEM_LD32(tmem_O + lane_base + c * 32, raw);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) raw[i] = __float_as_uint(__uint_as_float(raw[i]) * alpha);
            MMDIT_TMEM_ST32(tmem_O + lane_base + c * 32, raw);
          }
          tmem_wait_st();
        }
        l_run *= alpha;
        m_run = m_new;
      }
      float lsum = 0.f;
      uint32_t pk[kAttnBN / 2];
#pragma unroll
      for (int c = 0; c < kAttnBN / 2; ++c) {
        const float p0 = ex2_approx(fmaf(s[2 * c], sl2, -m_run));
        const float p1 = ex2_approx(fmaf(s[2 * c + 1], sl2, -m_run));
        lsum += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l_run += lsum;
      // P row r into the two 64-key halves, 16-byte chunks swizzled by r & 7.
#pragma unroll
      for (int kh = 0; kh < 2; ++kh) {
        uint8_t* rowp = sP + kh * kHalf + r * 128;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const int base = kh * 32 + ch * 4;
          *reinterpret_cast<uint4*>(rowp + ((ch ^ (r & 7)) << 4)) =
              make_uint4(pk[base], pk[base + 1], pk[base + 2], pk[base + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok && mbar_wait(pv_done, (nkv - 1) & 1, abort_flag, p.status, ST_TIMEOUT_SOFTMAX)) {
      tc_fence_after();
      const float inv_l = 1.0f / l_run;
      const int row = q0 + r;
      uint16_t* dst = p.out + ((long long)b * p.L + row) * p.out_ld + h * HD;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t raw[32];
        MMDIT_TMEM_LD32(tmem_O + lane_base + c * 32, raw);
        tmem_wait_ld();
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(raw[i]) * inv_l;
        if (row < p.L) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            d4[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                               pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
        }
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

template <int HD>
cudaError_t launch_attn_hd(const CUtensorMap& tmQK, const CUtensorMap& tmV, const AttnParams& p, cudaStream_t s) {
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)AttnSmem<HD>::total);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  dim3 grid(p.n_q_tiles, p.H, p.B);
  launch_begin(KID_ATTENTION, s);
  attn_fwd_kernel<HD><<<grid, kAttnThreads, AttnSmem<HD>::total, s>>>(tmQK, tmV, p);
  launch_end(s);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const CUtensorMap& tmQK, const CUtensorMap& tmV, const AttnParams& p, int d_head,
                             cudaStream_t s) {
  if (d_head == 128) return launch_attn_hd<128>(tmQK, tmV, p, s);
  return launch_attn_hd<64>(tmQK, tmV, p, s);
}

}  // namespace mmdit
