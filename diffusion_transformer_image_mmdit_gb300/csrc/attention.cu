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
// MMA shapes: S = Q K^T is M=128, N=128 keys, K=d (both operands K-major
// in shared memory, 128-byte swizzle); O += P V is M=128, N=d, K=128 keys
// with P read from tensor memory.  The running max lives in the log2
// domain; O is rescaled in TMEM only when the running max grows by more
// than 16 (a factor 2^16), which stays exact because the same reference is
// used for the numerator and the row sum: P entries stay below 2^16 (bf16
// keeps its relative precision there) and the fp32 sums far from overflow.
//
// Work schedule (persistent, one CTA per SM).  A work unit is a pair of
// query tiles (256 rows) of one (sample, head) over all n_kv KV tiles.  CTA
// c of G runs whole units c, c + G, ... for `dp_rounds` rounds; the units
// left after those rounds (between G and 2G of them) form the tail, whose KV
// steps (numbered unit by unit) are cut into G equal contiguous ranges, one
// per CTA.  Every CTA thus does the same number of KV steps to within one,
// where one unit per CTA launched as a grid left the SMs of the last partial
// wave idle.  A range is at least n_kv steps long, so a tail unit is split
// at most once, at the boundary between CTAs c and c + 1: part A (its first
// KV tiles) is the last item of CTA c, part B (the rest) the first tail item
// of CTA c + 1.  Each part writes its unnormalised O rows with their running
// max and sum (fp32) to its slot in global memory and counts itself on the
// unit's counter; the part that arrives second reads the other slot, merges
// the two with the usual rescaling, O = (2^(m_A - m) O_A + 2^(m_B - m) O_B) /
// (2^(m_A - m) l_A + 2^(m_B - m) l_B) with m = max(m_A, m_B), and stores the
// result, then sets the counter back to zero, so the counters need clearing
// only before the first launch over a merge area.  Neither part waits for the
// other.  With no more units than SMs
// each CTA runs one unit, and a launch given no merge area runs every unit
// whole, round-robin.  Consecutive items of a CTA overlap: the next item's K
// tile and Q tiles load while the current item's last P V MMAs and epilogue
// run.
#include <mutex>

#include "common.cuh"

namespace mmdit {

namespace {

constexpr uint32_t kHalf = 128 * 128;  // one 128-row x 128-byte swizzled half tile
constexpr float kRescaleThreshold = 16.0f;

// Roles (two query tiles per CTA, K/V tiles shared):
//   warps 0-3   softmax of tile 0; warps 4-7 softmax of tile 1 (one query
//               row per thread, 208 registers each after setmaxnreg so a
//               whole 128-score row stays in registers).  P goes back to
//               TMEM in two halves, each with its own barrier, so P V(j)
//               starts on keys 0..63 while keys 64..127 are exponentiated.
//               At the end of an item the warps read O out of TMEM (then
//               hand the columns back), and store O / l through their own
//               4 KB of shared memory with TMA tile stores, or write and
//               merge the partial result of a split unit.
//   warp 8      TMA: per item its first K tile, the two Q tiles (each once
//               the previous item's last S MMA of that tile has completed),
//               then V^T(j) and K(j + 1) tiles (the order their ring slots
//               free up and the MMAs need them), 2-stage rings.
//   warp 9      TMEM (S0 | S1 | O0 | O1, 128 columns each) and the MMAs, in
//               the order S0(0), S1(0), then per j: PV0(j), S0(j+1), PV1(j),
//               S1(j+1), so the tensor pipe works on one tile while the
//               other tile's softmax runs.  P(j) is written by the softmax
//               over the first 64 columns of S(j) as packed bf16 and read by
//               the P V MMA straight from TMEM; S(j+1) reuses the columns
//               only after PV(j), which precedes it in the MMA issue order.
//               The tensor pipe accepts only a few MMAs ahead of the one it
//               executes, so the issuing warp runs close behind it: every
//               wait it makes (about 175 cycles even on a completed phase),
//               every branch around an MMA group and every extra commit
//               shows up as idle tensor cycles.  The steady-state loop is
//               therefore straight-line (the last KV tile of an item is
//               peeled off), each wait (P halves, K(j+1), V(j+1)) sits
//               behind at least four queued MMAs that cover it, and the K
//               ring slot is released by the softmax warps of tile 1 (they
//               see S1(j) complete) instead of by a second commit.
//   warps 10-11 idle (they complete the third warpgroup, which gives its
//               registers to the softmax warpgroups).
// Barrier phases run on across items: ring stages and the per-step
// barriers follow a KV-step count kept by every role, the per-item barriers
// (Q tiles, P V done, O drained) the item count.
constexpr int kAttn2Threads = 384;
// Register split (setmaxnreg): launched at 168 per thread (384 x 168 = 64512);
// warpgroup 2 drops to 88 and the two softmax warpgroups rise to 208:
// 128 x 88 + 256 x 208 = 64512.  A softmax thread holds a 128-score row
// and 64 packed P words; the MMA warp's unrolled issue loop needs about 88.
constexpr uint32_t kRegsSoftmax = 208;
constexpr uint32_t kRegsControl = 88;
constexpr uint32_t kStageO = 4096;  // a softmax warp's O staging block: 32 rows x 64 columns bf16

template <int HD>
struct Attn2Smem {
  static constexpr uint32_t QT = (HD / 64) * kHalf;  // one 128-row Q tile
  static constexpr uint32_t K = (HD / 64) * kHalf;
  static constexpr uint32_t V = 2 * HD * 128;
  static constexpr uint32_t total = 1024 + 2 * QT + 2 * K + 2 * V + 8 * kStageO + 256;
};
static_assert(Attn2Smem<128>::total <= 232448, "attention shared memory above the 227 KB a CTA can have");

struct AttnItem {
  int u, jb, je;  // unit, KV tiles [jb, je)
};

// The items of this CTA, in order (identical in every role).
struct AttnWork {
  int c, G, nkv, round, rounds, units, base;
  long long s, s1;  // this CTA's range of tail KV steps
  __device__ explicit AttnWork(const AttnParams& p) {
    c = (int)blockIdx.x;
    G = (int)gridDim.x;
    nkv = p.n_kv_tiles;
    round = 0;
    rounds = p.dp_rounds;
    units = p.n_units;
    base = rounds * G;
    const long long T = (long long)p.tail_units * nkv;
    s = T * c / G;
    s1 = T * (c + 1) / G;
  }
  __device__ bool next(AttnItem& it) {
    while (round < rounds) {
      const int u = round++ * G + c;
      if (u < units) {
        it.u = u, it.jb = 0, it.je = nkv;
        return true;
      }
    }
    if (s >= s1) return false;
    const long long uo = s / nkv;
    const int jb = (int)(s - uo * nkv);
    const long long left = s1 - s;
    const int je = left < (long long)(nkv - jb) ? jb + (int)left : nkv;
    it.u = base + (int)uo, it.jb = jb, it.je = je;
    s += je - jb;
    return true;
  }
};

template <int HD>
__global__ void __launch_bounds__(kAttn2Threads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmO, const __grid_constant__ AttnParams p) {
  using SM = Attn2Smem<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + 2 * SM::QT;
  uint8_t* sV = sK + 2 * SM::K;
  uint8_t* sO = sV + 2 * SM::V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sO + 8 * kStageO);
  const uint32_t q_full0 = smem_u32(bars + 0);    // [2] per tile: Q tile loaded (once per item)
  const uint32_t k_full0 = smem_u32(bars + 2);    // [2] per stage
  const uint32_t v_full0 = smem_u32(bars + 4);    // [2] per stage
  const uint32_t k_empty0 = smem_u32(bars + 6);   // [2] per stage: freed once S1 of the K tile has completed
  const uint32_t s_full0 = smem_u32(bars + 8);    // [2] per tile
  const uint32_t p_full0 = smem_u32(bars + 10);   // [2] per tile
  const uint32_t pv_done0 = smem_u32(bars + 12);  // [2] per tile: the item's last P V has completed
  const uint32_t v_empty0 = smem_u32(bars + 14);  // [2] per stage: freed after both P V MMAs of the V tile
  const uint32_t mma_done = smem_u32(bars + 16);  // after a time-out: every issued MMA has completed
  const uint32_t p_half0 = smem_u32(bars + 17);   // [2] per tile: P over keys 0..63 written
  const uint32_t q_empty0 = smem_u32(bars + 19);  // [2] per tile: the item's last S MMA of the tile has completed
  const uint32_t o_free0 = smem_u32(bars + 21);   // [2] per tile: O read out of TMEM by the tile's softmax warps
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 23);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int D = p.H * HD;
  const int nkv = p.n_kv_tiles;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(q_full0 + 8 * i, 1);
      mbar_init(q_empty0 + 8 * i, 1);
      mbar_init(k_full0 + 8 * i, 1);
      mbar_init(v_full0 + 8 * i, 1);
      mbar_init(k_empty0 + 8 * i, 1);
      mbar_init(v_empty0 + 8 * i, 1);
      mbar_init(s_full0 + 8 * i, 1);
      mbar_init(p_full0 + 8 * i, 4);
      mbar_init(p_half0 + 8 * i, 4);
      mbar_init(pv_done0 + 8 * i, 1);
      mbar_init(o_free0 + 8 * i, 4);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmQK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    const int t = warp >> 2;
    const int quad = warp & 3;
    const int wid = warp;  // t * 4 + quad
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * 128;
    const uint32_t tO = tmem + lane_base + 256 + t * 128;
    const uint32_t s_full = s_full0 + 8 * t, p_full = p_full0 + 8 * t, p_half = p_half0 + 8 * t;
    const uint32_t pv_done = pv_done0 + 8 * t, o_free = o_free0 + 8 * t;
    uint8_t* stg = sO + wid * kStageO;
    const float sl2 = p.scale_log2;
    AttnWork work(p);
    AttnItem I;
    uint32_t g = 0, it = 0;  // KV steps and items done
    bool ok = true;
    while (ok && work.next(I)) {
      const int n = I.je - I.jb;
      float m_run = -INFINITY, l_run = 0.f;
#pragma unroll 1
      for (int jj = 0; jj < n; ++jj) {
        const uint32_t gj = g + (uint32_t)jj;
        if (!mbar_wait_warp(s_full, gj & 1, abort_flag, p.status, ST_TIMEOUT_SOFTMAX)) { ok = false; break; }
        tc_fence_after();
        // S1(j) has completed, and S0(j) before it: the K(j) ring slot is free
        if (t == 1 && quad == 0 && lane == 0) mbar_arrive(k_empty0 + 8 * (gj & 1));
        const int kv0 = (I.jb + jj) * kAttnBN;
        float sv[kAttnBN];
        {
          uint32_t raw[kAttnBN];
#pragma unroll
          for (int c = 0; c < kAttnBN / 32; ++c) MMDIT_TMEM_LD32(tS + c * 32, (raw + c * 32));
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < kAttnBN; ++c) sv[c] = __uint_as_float(raw[c]);
        }
        if (kv0 + kAttnBN > p.L) {
#pragma unroll
          for (int c = 0; c < kAttnBN; ++c)
            if (kv0 + c >= p.L) sv[c] = -INFINITY;
        }
        // row max: 8 independent chains of three-input max over columns
        // 8..119 in pairs of 8, then columns 120..127
        float mx8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = sv[i];
#pragma unroll
        for (int c = 8; c + 16 <= kAttnBN; c += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i) mx8[i] = fmax3(mx8[i], sv[c + i], sv[c + 8 + i]);
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], sv[kAttnBN - 8 + i]);
        const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
        const float m_new = fmaxf(m_run, mx * sl2);
        // P V(j - 1) has completed here: S(j) was issued after it and the
        // commit behind s_full covers every earlier MMA of the issuing thread.
        // So O may be rescaled, and P(j) may overwrite P(j - 1), without a
        // further wait.
        // Lazy rescale: the TMEM accesses are warp-wide, so the warp rescales
        // when any of its rows needs it (alpha = 1, an exact no-op, for the
        // others).  The item's first P V overwrites O, so its first step has
        // nothing to rescale.
        const bool grow = m_new > m_run + kRescaleThreshold;
        if (__any_sync(0xffffffffu, grow)) {
          const float alpha = grow ? ex2_approx(m_run - m_new) : 1.0f;
          if (jj > 0) {
#pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
              uint32_t raw[32];
              MMDIT_TMEM_LD32(tO + c * 32, raw);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) raw[i] = __float_as_uint(__uint_as_float(raw[i]) * alpha);
              MMDIT_TMEM_ST32(tO + c * 32, raw);
            }
            tmem_wait_st();
          }
          if (grow) {
            l_run *= alpha;
            m_run = m_new;
          }
        }
        // exponentials on column pairs (f32x2 arithmetic for the argument and the
        // sums), row sum in 4 packed partial sums, bf16 P over the first 64
        // columns of S.  Every exponential is a MUFU ex2: at 32 results per
        // cycle per SM it takes fewer issue slots than a polynomial on the FMA
        // pipe, and the softmax is issue-bound.
        const uint64_t sl2x2 = f2_pack(sl2, sl2), negm2 = f2_pack(-m_run, -m_run);
        uint64_t ls2[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) ls2[i] = f2_pack(0.f, 0.f);
        uint32_t pk[kAttnBN / 2];
#pragma unroll
        for (int c = 0; c < kAttnBN / 2; ++c) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(sv[2 * c], sv[2 * c + 1]), sl2x2, negm2), x0, x1);
          const uint64_t p2 = f2_pack(ex2_approx(x0), ex2_approx(x1));
          ls2[c & 3] = f2_add(ls2[c & 3], p2);
          float p0, p1;
          f2_unpack(p2, p0, p1);
          pk[c] = pack_bf16x2(p0, p1);
          // P over keys 0..63 is complete after pair 31: it is stored then,
          // and handed over 8 pairs later (the store's latency overlaps those
          // pairs), so that P V(j) starts on those keys while the other half
          // is computed.
          if (c == kAttnBN / 4 - 1) MMDIT_TMEM_ST32(tS, pk);
          if (c == kAttnBN / 4 + 7) {
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_half);
          }
        }
        float ls[2];
        f2_unpack(f2_add(f2_add(ls2[0], ls2[1]), f2_add(ls2[2], ls2[3])), ls[0], ls[1]);
        MMDIT_TMEM_ST32(tS + 32, (pk + 32));
        l_run += ls[0] + ls[1];
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
      }
      if (!ok || !mbar_wait_warp(pv_done, it & 1, abort_flag, p.status, ST_TIMEOUT_SOFTMAX)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // O of this warp's 32 rows into registers; the columns go back to the
      // MMA warp at once (the next item's first P V overwrites them).
      float o[HD];
      {
        uint32_t raw[HD];
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) MMDIT_TMEM_LD32(tO + c * 32, (raw + c * 32));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < HD; ++c) o[c] = __uint_as_float(raw[c]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);

      const int pair = I.u % p.n_pairs;
      const int bh = I.u / p.n_pairs;
      const int h = bh % p.H, b = bh / p.H;
      bool store = true;
      if (I.jb > 0 || I.je < nkv) {
        // Part of a split unit: A (keys from 0) is the last item of CTA c,
        // B (keys up to the end) the first tail item of CTA c + 1; boundary c
        // names the unit.  Slot layout per warp: O as [HD / 4][32 lanes]
        // float4 (coalesced rows of 512 bytes), then m[32], l[32].
        const int part = I.jb > 0 ? 1 : 0;
        const int bound = (int)blockIdx.x - part;
        constexpr int kSlot = 32 * HD + 64;
        float* own = p.part + (size_t)((bound * 2 + part) * 8 + wid) * kSlot;
        const float* oth = p.part + (size_t)((bound * 2 + (part ^ 1)) * 8 + wid) * kSlot;
        float4* own4 = reinterpret_cast<float4*>(own);
#pragma unroll
        for (int k = 0; k < HD / 4; ++k)
          __stcg(own4 + k * 32 + lane, make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]));
        __stcg(own + 32 * HD + lane, m_run);
        __stcg(own + 32 * HD + 32 + lane, l_run);
        __threadfence();
        __syncwarp();
        int second = 0;
        if (lane == 0) second = atomicAdd(p.cnt + bound * 8 + wid, 1) != 0;
        second = __shfl_sync(0xffffffffu, second, 0);
        if (!second) {
          store = false;  // the other part, still running, merges and stores
        } else {
          // both parts have counted: the counter goes back to zero for the
          // next launch that uses this merge area
          if (lane == 0) p.cnt[bound * 8 + wid] = 0;
          __threadfence();
          const float m_o = __ldcg(oth + 32 * HD + lane);
          const float l_o = __ldcg(oth + 32 * HD + 32 + lane);
          const float m = fmaxf(m_run, m_o);
          const float a = ex2_approx(m_run - m), c = ex2_approx(m_o - m);
          l_run = a * l_run + c * l_o;
          const float4* oth4 = reinterpret_cast<const float4*>(oth);
#pragma unroll
          for (int k = 0; k < HD / 4; ++k) {
            const float4 w = __ldcg(oth4 + k * 32 + lane);
            o[4 * k] = fmaf(a, o[4 * k], c * w.x);
            o[4 * k + 1] = fmaf(a, o[4 * k + 1], c * w.y);
            o[4 * k + 2] = fmaf(a, o[4 * k + 2], c * w.z);
            o[4 * k + 3] = fmaf(a, o[4 * k + 3], c * w.w);
          }
        }
      }
      if (store) {
        // O / l as bf16 through this warp's staging block, 64 columns at a
        // time, in the 128-byte-swizzled layout of the output tensor map --
        // row `lane` at a 128-byte pitch, 16-byte chunk i at position
        // i ^ (lane % 8) -- written out by lane 0 with TMA tile stores (rows
        // at or beyond L are clipped by the tensor map).  A warp's 16-byte
        // shared stores take 4 wavefronts each, where direct row-per-thread
        // global stores touched 32 scattered sectors per instruction.
        const float inv_l = 1.0f / l_run;
        const int row0 = pair * (2 * kAttnBM) + t * kAttnBM + quad * 32;
        uint8_t* rowp = stg + lane * 128;
#pragma unroll
        for (int hf = 0; hf < HD / 64; ++hf) {
          if (lane == 0) bulk_wait_group_read0();  // the previous store has read the block
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float* v = o + hf * 64 + 8 * i;
            *reinterpret_cast<uint4*>(rowp + ((i ^ (lane & 7)) << 4)) =
                make_uint4(pack_bf16x2(v[0] * inv_l, v[1] * inv_l), pack_bf16x2(v[2] * inv_l, v[3] * inv_l),
                           pack_bf16x2(v[4] * inv_l, v[5] * inv_l), pack_bf16x2(v[6] * inv_l, v[7] * inv_l));
          }
          fence_proxy_async_smem();  // the shared stores are visible to the TMA unit
          __syncwarp();
          if (lane == 0 && row0 < p.L) {
            tma_store_3d(&tmO, smem_u32(stg), h * HD + hf * 64, row0, b);
            bulk_commit_group();
          }
        }
      }
      g += (uint32_t)n;
      ++it;
    }
    if (lane == 0) bulk_wait_group_read0();  // the staging block has been read before the CTA exits
    __syncwarp();
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
    if (warp == 8) {
      if (lane == 0) {
        // Loads in the order the MMAs need them: per item K(first), the Q
        // tiles, then V(j) (for P V0(j)) before K(j + 1) (for S0(j + 1),
        // issued after P V0(j)).  This is also the order in which their slots
        // free up: V(j)'s after P V1(j - 2), K(j + 1)'s after S1(j - 1), Q
        // tile t's after the previous item's last S MMA of tile t.
        uint32_t n_k = 0, n_v = 0, n_item = 0;  // loads issued (ring counters, and for the drain after a time-out)
        uint32_t n_q[2] = {0, 0};
        int h = 0, b = 0;
        auto load_k = [&](int j) -> bool {
          const uint32_t st = n_k & 1;
          if (!mbar_wait(k_empty0 + 8 * st, ((n_k >> 1) & 1) ^ 1, abort_flag, p.status, ST_TIMEOUT_PRODUCER))
            return false;
          ++n_k;
          mbar_expect_tx(k_full0 + 8 * st, SM::K);
#pragma unroll
          for (int hf = 0; hf < HD / 64; ++hf)
            tma_load_3d(smem_u32(sK + st * SM::K + hf * kHalf), &tmQK, k_full0 + 8 * st, D + h * HD + hf * 64,
                        j * kAttnBN, b);
          return true;
        };
        auto load_v = [&](int j) -> bool {
          const uint32_t st = n_v & 1;
          if (!mbar_wait(v_empty0 + 8 * st, ((n_v >> 1) & 1) ^ 1, abort_flag, p.status, ST_TIMEOUT_PRODUCER))
            return false;
          ++n_v;
          mbar_expect_tx(v_full0 + 8 * st, SM::V);
#pragma unroll
          for (int kh = 0; kh < 2; ++kh)
            tma_load_3d(smem_u32(sV + st * SM::V + kh * (HD * 128)), &tmV, v_full0 + 8 * st, j * kAttnBN + kh * 64,
                        h * HD, b);
          return true;
        };
        AttnWork work(p);
        AttnItem I;
        bool okp = true;
        while (okp && work.next(I)) {
          const int pair = I.u % p.n_pairs;
          const int bh = I.u / p.n_pairs;
          h = bh % p.H, b = bh / p.H;
          okp = load_k(I.jb);
          for (int t = 0; okp && t < 2; ++t) {
            if (n_item > 0 &&
                !mbar_wait(q_empty0 + 8 * t, (n_item - 1) & 1, abort_flag, p.status, ST_TIMEOUT_PRODUCER)) {
              okp = false;
              break;
            }
            ++n_q[t];
            mbar_expect_tx(q_full0 + 8 * t, SM::QT);
#pragma unroll
            for (int hf = 0; hf < HD / 64; ++hf)
              tma_load_3d(smem_u32(sQ + t * SM::QT + hf * kHalf), &tmQK, q_full0 + 8 * t, h * HD + hf * 64,
                          pair * (2 * kAttnBM) + t * kAttnBM, b);
          }
          for (int j = I.jb; okp && j < I.je; ++j) okp = load_v(j) && (j + 1 >= I.je || load_k(j + 1));
          ++n_item;
        }
        if (*abort_flag) {
          // After a time-out anywhere in the CTA: wait (bounded) until every
          // copy still in flight into this CTA's shared memory has landed
          // (the last Q load of each tile, and the last two K and V tiles,
          // one per ring stage) before the CTA frees its resources and exits.
          constexpr unsigned long long kDrainNs = 100000000ull;
          for (int t = 0; t < 2; ++t)
            if (n_q[t] > 0) mbar_wait(q_full0 + 8 * t, (n_q[t] - 1) & 1, nullptr, nullptr, 0, kDrainNs);
          for (uint32_t j = n_k > 2 ? n_k - 2 : 0; j < n_k; ++j)
            mbar_wait(k_full0 + 8 * (j & 1), (j >> 1) & 1, nullptr, nullptr, 0, kDrainNs);
          for (uint32_t j = n_v > 2 ? n_v - 2 : 0; j < n_v; ++j)
            mbar_wait(v_full0 + 8 * (j & 1), (j >> 1) & 1, nullptr, nullptr, 0, kDrainNs);
        }
      }
    } else if (warp == 9) {
      // The whole warp runs the issue loop (warp-uniform operands); the
      // elected lane issues the MMAs and commits.
      const uint32_t leader = elect_one_sync();
      const uint32_t idesc_s = idesc_bf16(128, kAttnBN);
      const uint32_t idesc_o = idesc_bf16(128, HD);
      // Descriptors of Q tile 0 and of ring stage 0 are built once; an MMA
      // adds the tile / stage / K-step offset in 16-byte units to the start
      // address field (bits 0-13, which holds every shared address < 256 KB).
      const uint64_t dQ0 = sdesc_k128(smem_u32(sQ));
      const uint64_t dK0 = sdesc_k128(smem_u32(sK));
      const uint64_t dV0 = sdesc_k128(smem_u32(sV));
      auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
        return mbar_wait_warp(bar, parity, abort_flag, p.status, ST_TIMEOUT_MMA);
      };
      // S(t, g) = Q_t K(g)^T (kS = d / 16 steps of K = 16) and
      // O_t (+)= P_t(g) V(g) (8 steps: 128 keys), MMAs k0..k1-1 of those
      // steps; g counts KV steps over all items (it selects the ring stage).
      // Operand selection is arithmetic, not a branch.
      constexpr int kS = HD / 16;
      auto mma_s = [&](int t, uint32_t g, int k0, int k1) {
        const uint64_t aQ = dQ0 + (uint64_t)(t * (SM::QT >> 4));
        const uint64_t bK = dK0 + (uint64_t)((g & 1) * (SM::K >> 4));
        const uint32_t dS = tmem + t * 128;
#pragma unroll
        for (int k = k0; k < k1; ++k) {
          const uint32_t off = ((k >> 2) * kHalf + (k & 3) * 32) >> 4;
          umma_bf16_if(leader, dS, aQ + off, bK + off, idesc_s, k > 0 ? 1u : 0u);
        }
      };
      auto mma_pv = [&](int t, uint32_t g, uint32_t acc0, int k0, int k1) {
        const uint64_t bV = dV0 + (uint64_t)((g & 1) * (SM::V >> 4));
        const uint32_t dO = tmem + 256 + t * 128, aP = tmem + t * 128;
#pragma unroll
        for (int k = k0; k < k1; ++k) {
          const uint32_t off = ((k >> 2) * (HD * 128) + (k & 3) * 32) >> 4;
          umma_bf16_ta_if(leader, dO, aP + k * 8, bV + off, idesc_o, k > 0 ? 1u : acc0);
        }
      };
      // After a failed wait the loop still issues the MMAs of that step (all
      // operands lie inside this CTA's shared and tensor memory) and stops at
      // the next loop test: no branch sits between the waits and the MMAs.
      AttnWork work(p);
      AttnItem I;
      uint32_t g = 0, it = 0;
      bool ok = true;
      while (ok && work.next(I)) {
        const int n = I.je - I.jb;
        const uint32_t ph_it = it & 1;
        ok = wait(q_full0, ph_it) && wait(k_full0 + 8 * (g & 1), (g >> 1) & 1);
        tc_fence_after();
        mma_s(0, g, 0, kS);
        umma_commit_if(leader, s_full0);
        if (n == 1) umma_commit_if(leader, q_empty0);
        ok = wait(q_full0 + 8, ph_it) && ok;
        tc_fence_after();
        mma_s(1, g, 0, kS / 2);
        ok = wait(v_full0 + 8 * (g & 1), (g >> 1) & 1) && ok;
        tc_fence_after();
        mma_s(1, g, kS / 2, kS);
        umma_commit_if(leader, s_full0 + 8);
        if (n == 1) umma_commit_if(leader, q_empty0 + 8);
        if (it > 0) {
          // the previous item's O columns have been read out (the first P V
          // of this item overwrites them)
          ok = wait(o_free0, ph_it ^ 1) && ok;
          ok = wait(o_free0 + 8, ph_it ^ 1) && ok;
          tc_fence_after();
        }
        int jj = 0;
#pragma unroll 1
        for (; ok && jj + 1 < n; ++jj) {
          const uint32_t gj = g + (uint32_t)jj, gn = gj + 1;
          const uint32_t st1 = gn & 1, ph1 = (gn >> 1) & 1;
          const uint32_t acc0 = jj > 0 ? 1u : 0u;
          ok = wait(p_half0, gj & 1);  // P0(j) over keys 0..63
          tc_fence_after();
          mma_pv(0, gj, acc0, 0, 4);
          ok = wait(p_full0, gj & 1) && ok;  // P0(j) over keys 64..127
          tc_fence_after();
          mma_pv(0, gj, acc0, 4, 8);
          ok = wait(k_full0 + 8 * st1, ph1) && ok;  // K(j + 1), for S0(j + 1)
          tc_fence_after();
          mma_s(0, gn, 0, kS);
          umma_commit_if(leader, s_full0);
          if (jj + 2 == n) umma_commit_if(leader, q_empty0);  // the item's last S0
          ok = wait(p_half0 + 8, gj & 1) && ok;
          tc_fence_after();
          mma_pv(1, gj, acc0, 0, 4);
          ok = wait(p_full0 + 8, gj & 1) && ok;
          tc_fence_after();
          mma_pv(1, gj, acc0, 4, 8);
          umma_commit_if(leader, v_empty0 + 8 * (gj & 1));  // P V0(j) and P V1(j) have read V(j)
          mma_s(1, gn, 0, kS / 2);
          ok = wait(v_full0 + 8 * st1, ph1) && ok;  // V(j + 1), for P V0(j + 1)
          tc_fence_after();
          mma_s(1, gn, kS / 2, kS);
          umma_commit_if(leader, s_full0 + 8);
          if (jj + 2 == n) umma_commit_if(leader, q_empty0 + 8);  // the item's last S1
        }
        if (ok) {  // the item's last KV tile
          const uint32_t gj = g + (uint32_t)jj;
          const uint32_t acc0 = jj > 0 ? 1u : 0u;
          ok = wait(p_half0, gj & 1);
          tc_fence_after();
          mma_pv(0, gj, acc0, 0, 4);
          ok = wait(p_full0, gj & 1) && ok;
          tc_fence_after();
          mma_pv(0, gj, acc0, 4, 8);
          umma_commit_if(leader, pv_done0);  // for the final O / l
          ok = wait(p_half0 + 8, gj & 1) && ok;
          tc_fence_after();
          mma_pv(1, gj, acc0, 0, 4);
          ok = wait(p_full0 + 8, gj & 1) && ok;
          tc_fence_after();
          mma_pv(1, gj, acc0, 4, 8);
          umma_commit_if(leader, v_empty0 + 8 * (gj & 1));
          umma_commit_if(leader, pv_done0 + 8);
        }
        g += (uint32_t)n;
        ++it;
      }
      if (*abort_flag) {
        // every MMA this warp issued (they read shared memory and write the
        // tensor memory about to be freed) completes first
        umma_commit_if(leader, mma_done);
        mbar_wait_warp(mma_done, 0, nullptr, nullptr, 0);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int HD>
cudaError_t launch_attn2_hd(const CUtensorMap& tmQK, const CUtensorMap& tmV, const CUtensorMap& tmO,
                            const AttnParams& p_in, cudaStream_t s) {
  // shared-memory opt-in once per device, safe under concurrent first calls
  static std::once_flag once[64];
  static cudaError_t setup_err[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::call_once(once[dev], [&] {
    setup_err[dev] = cudaFuncSetAttribute(attn_fwd_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)Attn2Smem<HD>::total);
  });
  if (setup_err[dev] != cudaSuccess) return setup_err[dev];
  AttnParams p = p_in;
  p.n_pairs = (p.n_q_tiles + 1) / 2;
  p.n_units = p.n_pairs * p.H * p.B;
  if (p.n_units <= 0) return cudaSuccess;
  int G = num_sms();
  if (G > kAttnMaxCtas) G = kAttnMaxCtas;
  if (G > p.n_units) G = p.n_units;
  if (G < 1) return cudaErrorInvalidConfiguration;
  if (p.part && p.cnt && p.n_units > G) {
    // whole rounds, then the last one to two rounds' worth of units balanced
    p.dp_rounds = p.n_units / G - 1;
    p.tail_units = p.n_units - p.dp_rounds * G;
    if (!p.cnt_zero) {
      cudaError_t e = cudaMemsetAsync(p.cnt, 0, sizeof(int) * 8 * (size_t)G, s);
      if (e != cudaSuccess) return e;
    }
  } else {
    p.dp_rounds = (p.n_units + G - 1) / G;
    p.tail_units = 0;
  }
  launch_begin(KID_ATTENTION, s);
  attn_fwd_kernel<HD><<<G, kAttn2Threads, Attn2Smem<HD>::total, s>>>(tmQK, tmV, tmO, p);
  launch_end(s);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const CUtensorMap& tmQK, const CUtensorMap& tmV, const CUtensorMap& tmO,
                             const AttnParams& p, int d_head, cudaStream_t s) {
  if (d_head == 128) return launch_attn2_hd<128>(tmQK, tmV, tmO, p, s);
  return launch_attn2_hd<64>(tmQK, tmV, tmO, p, s);
}

}  // namespace mmdit
