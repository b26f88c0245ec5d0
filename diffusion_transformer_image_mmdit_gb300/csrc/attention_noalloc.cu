// joint_attention_fwd_noalloc: the joint-attention entry point for callers
// that cannot allocate device memory.
//
// joint_attention_fwd needs scratch for the normalised/rotated q and k and
// the transposed v, which its caller passes as a workspace.  Some callers
// cannot provide one: a plugin inside a host application that owns every
// device allocation and forbids its plugins from calling cudaMalloc, or code
// that must not risk the implicit device synchronisation cudaMalloc/cudaFree
// can cause.  This variant takes its scratch from a fixed, file-scope device
// array instead, so the call allocates nothing.
//
// Properties of the fixed scratch:
//  - kNoallocScratchBytes (48 MiB) per device, reserved for the lifetime of
//    the process on every GPU that loads this library; shapes needing more
//    are rejected with MMDIT_ERR_WORKSPACE before anything is launched.
//  - One array per device, shared by every call: calls whose work overlaps
//    on the GPU (for example on two streams at once) race on it.  Issue them
//    on one stream or serialise them.
//  - It keeps the previous call's contents.  Nothing needs clearing: every
//    scratch byte the attention kernel reads is written earlier in the same
//    call (the key extent of the V tensor map stops at L, so the padding
//    columns are never read).
//  - The first call on a device looks up the array's device address with
//    cudaGetSymbolAddress (with that device current) and caches it; make
//    that first call before any stream capture.
#include <atomic>

#include "elementwise.h"
#include "mmdit.h"
#include "mmdit_internal.h"

namespace mmdit {

namespace {

constexpr size_t kNoallocScratchBytes = 48ull << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch, per device, filled by the first call
// (threads racing on it compute the same address; the atomic publishes it).
void* scratch_address(int dev) {
  static std::atomic<void*> addr[64] = {};
  if (dev < 0 || dev >= 64) return nullptr;
  void* q = addr[dev].load(std::memory_order_acquire);
  if (!q) {
    if (cudaGetSymbolAddress(&q, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev].store(q, std::memory_order_release);
  }
  return q;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

}  // namespace mmdit

extern "C" int joint_attention_fwd_noalloc(const mmdit_shape_t* shape, const void* qkv, int qkv_row_stride,
                                           const float* const q_norm[2], const float* const k_norm[2],
                                           const float* cos_, const float* sin_, void* out, int out_row_stride,
                                           void* stream) {
  using namespace mmdit;
  // The public size query validates the shape; the scratch holds qk and vT
  // only (no merge area: the schedule here runs whole units).
  size_t need = 0;
  const int st = mmdit_workspace_size(shape, MMDIT_OP_ATTENTION, &need);
  if (st != MMDIT_OK) return st;
  {
    const size_t B = (size_t)shape->B;
    const size_t L = (size_t)shape->L_txt + (size_t)shape->grid_h * shape->grid_w + (size_t)shape->ref_h * shape->ref_w;
    const size_t D = (size_t)shape->D, Lp = (L + 7) / 8 * 8;
    need = ((B * L * 2 * D * 2 + 255) & ~size_t(255)) + B * D * Lp * 2;
  }
  if (need > kNoallocScratchBytes) return MMDIT_ERR_WORKSPACE;
  if (!qkv || !out) return MMDIT_ERR_ARG;
  if ((cos_ == nullptr) != (sin_ == nullptr)) return MMDIT_ERR_ARG;
  // the sequence is [text; target image; reference image] tokens, as in the workspace variant
  const int B = shape->B, Lt = shape->L_txt;
  const int L = shape->L_txt + shape->grid_h * shape->grid_w + shape->ref_h * shape->ref_w;
  const int D = shape->D, H = shape->H, d = shape->d_head;
  const int Lpad = (L + 7) / 8 * 8;
  if (qkv_row_stride < 3 * D || qkv_row_stride % 8 || out_row_stride < D || out_row_stride % 8)
    return MMDIT_ERR_SHAPE;
  if (!aligned16(qkv) || !aligned16(out)) return MMDIT_ERR_ALIGN;
  const float* gq0 = q_norm ? q_norm[0] : nullptr;
  const float* gq1 = q_norm ? q_norm[1] : nullptr;
  const float* gk0 = k_norm ? k_norm[0] : nullptr;
  const float* gk1 = k_norm ? k_norm[1] : nullptr;
  if (gq0 && (!gq1 || !gk0 || !gk1)) return MMDIT_ERR_ARG;

  // Same device checks as every other entry point (sm_103, the driver's
  // tensor-map encoder, the status word) before anything is launched.
  const int dc = device_check();
  if (dc != MMDIT_OK) return dc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MMDIT_ERR_CUDA;
  unsigned char* base = static_cast<unsigned char*>(scratch_address(dev));
  if (!base) return MMDIT_ERR_CUDA;

  // Same carving as the workspace variant: qk [B][L][2D], then vT [B][D][Lpad], 256-byte aligned.
  const size_t qk_bytes = (size_t)B * L * 2 * D * 2;
  uint16_t* qk = reinterpret_cast<uint16_t*>(base);
  uint16_t* vT = reinterpret_cast<uint16_t*>(base + ((qk_bytes + 255) & ~size_t(255)));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (launch_attn_prep(static_cast<const uint16_t*>(qkv), qkv_row_stride, B, L, Lt, H, d, gq0, gq1, gk0, gk1,
                       shape->eps_rms, cos_, sin_, qk, vT, Lpad, s) != cudaSuccess)
    return MMDIT_ERR_CUDA;
  // No merge area in the static scratch: the schedule runs whole units only.
  return run_attention_prepared(B, L, H, d, Lpad, qk, vT, static_cast<uint16_t*>(out), out_row_stride, nullptr,
                                nullptr, s);
}
