// Launchers of the bandwidth-bound kernels (elementwise.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mmdit {

// y[seg][i] = LN(x[seg*x_seg_rows + i]) (1 + scale[seg]) + shift[seg]; D % 256 == 0, D <= 4096.
// With q and qs: also the e4m3 rows of the bf16 result (row scale max|y| / 448 into qs[row], codes into
// q[row * D ..]); y may then be null (bf16 rows not stored).
struct LnJob {
  const float* x;
  long long x_seg_rows;
  int rows, n_seg;  // rows per segment (sample), segments
  const float* shift;
  const float* scale;  // modulation of segment s at shift / scale + s * mod_stride
  long long mod_stride;
  uint16_t* y;  // output row r (r = s * rows + i) at y + r * D
  uint8_t* q;
  float* qs;
};
struct LnJobs {
  LnJob job[2];
  int n0, n_total;  // rows of job 0; rows of both jobs
  float eps;
};
// One launch over one or two jobs with the same D and output kind (bf16 or e4m3 rows).
cudaError_t launch_ln_modulate_jobs(const LnJob* jobs, int n_jobs, int D, float eps, cudaStream_t st);
cudaError_t launch_ln_modulate(const float* x, long long x_seg_rows, int rows, int n_seg, int D, const float* shift,
                               const float* scale, long long mod_stride, float eps, uint16_t* y, cudaStream_t st,
                               uint8_t* q = nullptr, float* qs = nullptr);
cudaError_t launch_gemv(const void* W, bool i8, const float* wscale, const float* bias, const float* x, int B, int N,
                        int K, int act, float* y, cudaStream_t st);
// Many GEMVs sharing one input vector set x [B, K] (after the activation):
// job j computes out_j[b, n] = W_j act(x[b]) (* scale_j[n]) + bias_j[n] for
// n < N_j.  All jobs use the same weight type.
struct GemvJob {
  const void* W;
  const float* scale;
  const float* bias;
  float* out;
  int N;
  long long ldo;  // elements between the outputs of consecutive x rows (0: N)
};
cudaError_t launch_gemv_batched(const GemvJob* jobs, int n_jobs, bool i8, const float* x, int B, int K, int act,
                                cudaStream_t st);
// t_tab != null: t = t_scale * t_tab[*t_idx], read on the device.
cudaError_t launch_sinusoid(double t, int B, int dim, float* out, cudaStream_t st, const double* t_tab = nullptr,
                            const int* t_idx = nullptr, double t_scale = 1.0);
// Tokens: L_txt text, n_gen target image tokens on a grid_w-wide grid, then reference tokens on a ref_w-wide grid.
cudaError_t launch_rope_build(int L_txt, int grid_w, int n_gen, int ref_w, int L, const int axes[3], double theta,
                              int32_t* ids, float* cs,
                              float* sn, cudaStream_t st);
cudaError_t launch_rope_apply(uint16_t* x, long long rows, int L, int H, int d, int row_stride, const float* cs,
                              const float* sn, cudaStream_t st);
// sig_tab != null: dt = sig_tab[k + 1] - sig_tab[k], k = *sig_idx, read on the device.
cudaError_t launch_euler(float* x, const void* v, bool v_bf16, float dt, long long n, cudaStream_t st,
                         const double* sig_tab = nullptr, const int* sig_idx = nullptr);
// y += x (n floats).
cudaError_t launch_add(float* y, const float* x, long long n, cudaStream_t st);
// dst[i] = src[k * stride + i], i < n: step k's slice of a buffer computed for
// every step, k = *k_dev (device counter) when k_dev is given, else k_host.
cudaError_t launch_select_step(const float* src, long long stride, long long n, const int* k_dev, int k_host,
                               float* dst, cudaStream_t st);
// *c = value (add = false) or *c += value (add = true), one thread.
cudaError_t launch_counter(int* c, int value, bool add, cudaStream_t st);
cudaError_t launch_quantize(const void* w, bool w_bf16, int N, int K, int8_t* q, float* scale, cudaStream_t st);
cudaError_t launch_dequant_i8(const int8_t* q, uint16_t* out, long long n, cudaStream_t st);
// FP8 (e4m3) rows: x [rows, K] (row stride ld, bf16 or fp32) -> q [rows, K]
// (row stride qld) and scale [rows], s = max|row| / 448.
cudaError_t launch_quantize_f8(const void* x, bool x_bf16, long long rows, int K, long long ld, uint8_t* q,
                               long long qld, float* scale, cudaStream_t st);
cudaError_t launch_cast_bf16(const float* x, uint16_t* y, long long n, cudaStream_t st);
// Ulysses exchange layouts (bf16): pack src [rows][src_ld] (sections x groups x gc columns) into
// dst [groups][rows][sections][gc]; unpack src [groups][rows][gc] into dst [rows][dst_ld] (gc % 8 == 0).
cudaError_t launch_heads_pack(const uint16_t* src, long long rows, int src_ld, int sections, int groups, int gc,
                              uint16_t* dst, cudaStream_t st);
cudaError_t launch_heads_unpack(const uint16_t* src, long long rows, int groups, int gc, uint16_t* dst, int dst_ld,
                                cudaStream_t st);
cudaError_t launch_wait_selftest(unsigned long long limit_ns, unsigned* status, cudaStream_t st);
cudaError_t launch_attn_prep(const uint16_t* qkv, long long qkv_ld, int B, int L, int L_txt, int H, int d,
                             const float* gq0, const float* gq1, const float* gk0, const float* gk1, float eps,
                             const float* cs, const float* sn, uint16_t* qk, uint16_t* vT, long long vT_ld,
                             cudaStream_t st);

}  // namespace mmdit
