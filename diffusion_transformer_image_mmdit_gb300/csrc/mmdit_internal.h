// Internal declarations shared by the translation units of libmmdit.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mmdit {

// ----------------------------------------------------------------- GEMM
// Tile shape of the tcgen05 GEMM: 128 x 256 output tile per CTA (a CTA pair
// computes 256 x 256), K blocks of 64 bf16 (one 128-byte swizzle row).
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;

enum GemmMode : int {
  GM_STORE_BF16 = 0,  // out bf16, GELU on columns >= gelu_from
  GM_STORE_F32 = 1,   // out fp32
  GM_RESID = 2,       // resid fp32 += gate * value
  GM_QKV = 3,         // q,k: RMSNorm + RoPE -> qk; v -> transposed vT; rest: GELU -> aux
  GM_SWIGLU = 4,      // W rows [gate; up]: out bf16 = SiLU(gate) * up, N / 2 wide
};

// Rows are grouped in `n_seg` segments (samples) of M_seg rows each; the A
// operand's row r of segment s is read through a 3D tensor map (K, M_seg,
// n_seg).  Output row of (s, m) = s * out_seg_rows + out_row_off + m.
struct GemmParams {
  int M_seg, n_seg, N, K;
  int tiles_m, tiles_n, num_tiles, group_m;
  int mode;
  int gelu_from;
  int swiglu_up;  // GM_SWIGLU: row offset of the up half of W (= the output width)
  const float* bias;    // [N] or null
  const float* wscale;  // [N] or null (int8 or fp8 weights)
  const float* ascale;  // fp8 GEMM: scale of A row seg * ascale_seg_rows + m
  long long ascale_seg_rows;
  void* out;            // bf16 or fp32 output
  long long out_ld;
  long long out_seg_rows;
  int out_row_off;
  // GM_RESID (the update goes through GemmGroup::tmR; resid is its base)
  float* resid;
  long long resid_ld;
  long long resid_seg_rows;
  const float* gate;  // [n_seg][gate_seg_stride] or null
  long long gate_seg_stride;
  // GM_QKV
  int qkv_D;   // H * d_head
  int d_head;  // 64 or 128
  const float* gq;
  const float* gk;
  float eps;
  const float* rope_cos;  // [L, d_head/2]; table row = out_row_off + m
  const float* rope_sin;
  uint16_t* qk;  // [seg][out_seg_rows][qk_ld]: q at col n, k at col n
  long long qk_ld;
  uint16_t* vT;  // [seg][H*d][vT_ld]
  long long vT_ld;
  uint16_t* aux;  // rest columns n >= 3D -> aux[row][aux_col_off + n - 3D], GELU
  long long aux_ld;
  int aux_col_off;
  unsigned* status;
};

// One launch of the persistent GEMM serves up to two problems with the same
// tile shape (e.g. the text and image streams of a double block): tiles
// [0, tiles0) belong to problem 0, the rest to problem 1.
struct GemmGroup {
  CUtensorMap tmA[2];
  CUtensorMap tmB[2];
  CUtensorMap tmR[2];  // GM_RESID: the fp32 residual (cols N, rows M_seg, n_seg), 32 x 32 boxes, 128-byte swizzle
  GemmParams p[2];
  int n_prob;
  int tiles0;
  int total_tiles;
  int f8;  // both problems fp8 (e4m3 A and W, kind::f8f6f4) instead of bf16
};

// ----------------------------------------------------------------- attention
constexpr int kAttnBM = 128;  // queries per CTA
constexpr int kAttnBN = 128;  // keys per KV tile

constexpr int kAttnMaxCtas = 160;  // bound on the persistent attention grid (one CTA per SM)

struct AttnParams {
  int L, H, B, n_q_tiles, n_kv_tiles;
  float scale_log2;              // log2(e) / sqrt(d_head)
  unsigned* status;
  // Split-tail merge area (both null: whole units only, no split): per
  // boundary between consecutive CTAs, 8 counters (one per softmax warp) and
  // 2 x 8 slots of 32 x d_head + 64 floats; attn_merge_ctas(units)
  // boundaries at most.
  int* cnt;
  float* part;
  // Nonzero: the counters are known to be zero (the caller cleared them, and
  // every launch leaves them zero: the part that merges a split unit resets
  // the unit's counter), so the launcher does not clear them.
  int cnt_zero;
  // Set by the launcher: units (query-tile pairs x heads x samples), whole
  // rounds, and the tail units balanced over the grid.
  int n_pairs, n_units, dp_rounds, tail_units;
};
// Units of an attention launch: pairs of 128-row query tiles x heads x samples.
inline long long attn_units(int B, int L, int H) { return (long long)((L + 2 * kAttnBM - 1) / (2 * kAttnBM)) * H * B; }
// The persistent grid never exceeds the unit count, so neither do the boundaries.
inline size_t attn_merge_ctas(long long units) { return (size_t)(units < kAttnMaxCtas ? units : kAttnMaxCtas); }
inline size_t attn_merge_floats(int d_head, long long units) {
  return attn_merge_ctas(units) * 2 * 8 * (32 * (size_t)d_head + 64);
}

// ----------------------------------------------------------------- host helpers
unsigned* device_status_ptr();  // device address of the status word (current device)

// Kernel ids reported by the launch trace.
enum KernelId : int {
  KID_GEMM = 0,
  KID_ATTENTION,
  KID_LN_MODULATE,
  KID_GEMV,
  KID_SINUSOID,
  KID_ROPE_BUILD,
  KID_ROPE_APPLY,
  KID_EULER,
  KID_QUANTIZE,
  KID_DEQUANT,
  KID_CAST,
  KID_ATTN_PREP,
  KID_SELFTEST,
  KID_ADD,
  KID_COUNTER,
  KID_QUANTIZE_F8,
  KID_HEADS_PACK,
  KID_HEADS_UNPACK,
  KID_VT_TRANSPOSE,
  KID_SELECT_STEP,
  KID_COUNT
};
// Bracket every kernel launch: counts launches and, while a trace is on,
// records a CUDA event on the launch stream before and after the kernel.
void launch_begin(int kernel_id, cudaStream_t s);
void launch_end(cudaStream_t s);

// Encodes a 3D bf16 tensor map with a 64-element (128-byte) inner box and the
// 128-byte swizzle: dims (inner, rows, batch), byte strides of rows and batch.
bool make_tmap_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, uint64_t inner,
                  uint64_t rows, uint64_t batch, uint64_t row_stride_bytes, uint64_t batch_stride_bytes,
                  uint32_t box_inner, uint32_t box_rows, bool swizzle128);

// Launchers (return cudaError_t of the launch).
cudaError_t launch_gemm(const GemmGroup& g, cudaStream_t s);
// tmO: bf16 output [B][L][out_ld] (head h at column h*d), box 64 columns x 32
// rows, 128-byte swizzle.
cudaError_t launch_attention(const CUtensorMap& tmQK, const CUtensorMap& tmV, const CUtensorMap& tmO,
                             const AttnParams& p, int d_head, cudaStream_t s);
int num_sms();

// Status (an MMDIT_* code) of the current device for the kernels: sm_103,
// the tensor-map encoder of the driver found, the status word reachable.
int device_check();

// Joint attention over prepared operands: q and k rows in qk [B][L][2D]
// (normalised and rotated), v transposed in vT [B][D][Lpad]; writes out
// [B][L][out_ld] bf16.  merge_cnt / merge_part: the split-tail merge area
// (kAttnMaxCtas * 8 ints, attn_merge_floats(d_head) floats), or both null
// for a schedule of whole units only.  Returns an MMDIT_* status.
int run_attention_prepared(int B, int L, int H, int d_head, int Lpad, const uint16_t* qk, const uint16_t* vT,
                           uint16_t* out, long long out_ld, int* merge_cnt, float* merge_part, cudaStream_t st,
                           bool merge_cnt_zero = false);

}  // namespace mmdit
