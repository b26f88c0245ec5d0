// C ABI of libmmdit: argument checks, workspace carving, tensor maps and the
// kernel sequence of each block and of a whole denoising step.
#include <atomic>
#include <cmath>
#include <cstring>
#include <vector>

#include "elementwise.h"
#include "mmdit.h"
#include "mmdit_internal.h"

namespace mmdit {

// ----------------------------------------------------------------- process state
static __device__ unsigned g_status_word;
static std::atomic<long long> g_launches{0};

// Launch trace: a pool of CUDA events created by mmdit_trace_begin; while it
// is on, each launch records one event before and one after its kernel.
struct Trace {
  bool on = false;
  int cap = 0, n = 0;
  cudaEvent_t* ev = nullptr;  // 2 * cap
  int* ids = nullptr;         // cap
};
static Trace g_trace;

void launch_begin(int kernel_id, cudaStream_t s) {
  if (g_trace.on && g_trace.n < g_trace.cap) {
    g_trace.ids[g_trace.n] = kernel_id;
    cudaEventRecord(g_trace.ev[2 * g_trace.n], s);
  }
}

void launch_end(cudaStream_t s) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (g_trace.on && g_trace.n < g_trace.cap) {
    cudaEventRecord(g_trace.ev[2 * g_trace.n + 1], s);
    ++g_trace.n;
  }
}

static void trace_free() {
  if (g_trace.ev) {
    for (int i = 0; i < 2 * g_trace.cap; ++i) cudaEventDestroy(g_trace.ev[i]);
    delete[] g_trace.ev;
    delete[] g_trace.ids;
  }
  g_trace = Trace();
}

static int current_device() {
  int dev = 0;
  cudaGetDevice(&dev);
  return dev < 0 ? 0 : (dev > 63 ? 63 : dev);
}

// Per-device values looked up once.  Several host threads may race on the
// first lookup; each computes the same value, and the atomics make the
// publication well defined.
unsigned* device_status_ptr() {
  static std::atomic<unsigned*> ptrs[64] = {};
  const int dev = current_device();
  unsigned* q = ptrs[dev].load(std::memory_order_acquire);
  if (!q) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) == cudaSuccess) {
      q = static_cast<unsigned*>(p);
      ptrs[dev].store(q, std::memory_order_release);
    }
  }
  return q;
}

int num_sms() {
  static std::atomic<int> sms[64] = {};
  const int dev = current_device();
  int n = sms[dev].load(std::memory_order_relaxed);
  if (!n) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n = v > 0 ? v : 1;
    sms[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// 1 = sm_103, -1 = other device, 0 = unknown yet.
static int device_ok() {
  static std::atomic<int> ok[64] = {};
  const int dev = current_device();
  int k = ok[dev].load(std::memory_order_relaxed);
  if (!k) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return 0;
    k = (major == 10 && minor == 3) ? 1 : -1;
    ok[dev].store(k, std::memory_order_relaxed);
  }
  return k > 0;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool make_tmap_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, uint64_t inner,
                  uint64_t rows, uint64_t batch, uint64_t row_stride_bytes, uint64_t batch_stride_bytes,
                  uint32_t box_inner, uint32_t box_rows, bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  (void)elem_bytes;
  cuuint64_t dims[3] = {inner, rows, batch};
  cuuint64_t strides[2] = {row_stride_bytes, batch_stride_bytes};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ----------------------------------------------------------------- helpers
static inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static inline cudaStream_t S(void* s) { return reinterpret_cast<cudaStream_t>(s); }
static inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? MMDIT_OK : MMDIT_ERR_CUDA; }

#define MMDIT_TRY(expr)            \
  do {                             \
    const int _st = (expr);        \
    if (_st != MMDIT_OK) return _st; \
  } while (0)
#define MMDIT_CUDA(expr) MMDIT_TRY(cuda_status(expr))

// Bump allocator over the caller's workspace (or a size query with base == 0).
struct Carve {
  uint8_t* base;
  size_t off;
  template <class T>
  T* take(size_t n) {
    off = (off + 255) & ~size_t(255);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += n * sizeof(T);
    return p;
  }
};

struct Dims {
  int B, Lt, Li, L, Lpad, D, H, d, Dm;
  int Lg, Lr;  // image tokens per sample: Li = Lg target + Lr reference
  bool swiglu;  // SwiGLU MLP: the first MLP projection has 2 Dm rows [gate; up]
  bool f8;      // FP8 block GEMMs (MMDIT_F8W)
};

static int check_shape(const mmdit_shape_t* s, Dims* out) {
  if (!s) return MMDIT_ERR_ARG;
  if (s->B < 1 || s->L_txt < 0 || s->grid_h < 1 || s->grid_w < 1) return MMDIT_ERR_SHAPE;
  if (s->ref_h < 0 || s->ref_w < 0 || (s->ref_h == 0) != (s->ref_w == 0)) return MMDIT_ERR_SHAPE;
  if (s->D <= 0 || s->D % 256 || s->D > 4096) return MMDIT_ERR_SHAPE;
  if (s->d_head != 64 && s->d_head != 128) return MMDIT_ERR_SHAPE;
  if (s->H * s->d_head != s->D) return MMDIT_ERR_SHAPE;
  if (s->D_mlp <= 0 || s->D_mlp % 64) return MMDIT_ERR_SHAPE;
  const int a0 = s->rope_axes[0], a1 = s->rope_axes[1], a2 = s->rope_axes[2];
  if (a0 < 0 || a1 < 0 || a2 < 0 || (a0 | a1 | a2) & 1 || a0 + a1 + a2 != s->d_head) return MMDIT_ERR_SHAPE;
  if (s->w_dtype != MMDIT_BF16 && s->w_dtype != MMDIT_I8W && s->w_dtype != MMDIT_F8W) return MMDIT_ERR_ARG;
  if (s->mlp_act != MMDIT_MLP_GELU && s->mlp_act != MMDIT_MLP_SWIGLU) return MMDIT_ERR_ARG;
  if (s->mlp_act == MMDIT_MLP_SWIGLU && s->D_mlp % 128) return MMDIT_ERR_SHAPE;
  const long long Lg = (long long)s->grid_h * s->grid_w, Lr = (long long)s->ref_h * s->ref_w;
  const long long L = (long long)s->L_txt + Lg + Lr;
  if (L > (1 << 24)) return MMDIT_ERR_SHAPE;
  if (out) {
    out->B = s->B, out->Lt = s->L_txt, out->Li = (int)(Lg + Lr), out->L = (int)L;
    out->Lg = (int)Lg, out->Lr = (int)Lr;
    out->Lpad = (int)((L + 7) / 8 * 8);
    out->D = s->D, out->H = s->H, out->d = s->d_head, out->Dm = s->D_mlp;
    out->swiglu = s->mlp_act == MMDIT_MLP_SWIGLU;
    out->f8 = s->w_dtype == MMDIT_F8W;
    if (out->f8 && (s->D % 128 || s->D_mlp % 128)) return MMDIT_ERR_SHAPE;  // whole e4m3 K blocks
  }
  return MMDIT_OK;
}

int device_check() {
  if (!device_ok()) return MMDIT_ERR_UNSUPPORTED;
  if (!encode_fn()) return MMDIT_ERR_UNSUPPORTED;
  if (!device_status_ptr()) return MMDIT_ERR_CUDA;
  return MMDIT_OK;
}
static int check_device() { return device_check(); }

static bool lin_ok(const mmdit_linear_t& l, bool want_i8) {
  if (!l.w || !al16(l.w)) return false;
  if (l.b && !al16(l.b)) return false;
  if (want_i8 != (l.scale != nullptr)) return false;
  if (l.scale && !al16(l.scale)) return false;
  return true;
}

// ----------------------------------------------------------------- GEMM
// One problem of a GEMM launch: its tensor maps and epilogue parameters.
struct GemmProblem {
  CUtensorMap ta, tb, tr;
  GemmParams p;
  bool f8;
};

// A row r of segment s at A + (s * a_seg_rows + r) * a_ld (bf16 elements).
// Int8 weights are first widened into wdeq (exact), their scale goes to the epilogue.
// FP8 problems: p.ascale set by the caller (the per-row scales of the e4m3
// A); W is e4m3 with its per-channel scale in lin.scale; a K block is 128
// elements (128 bytes), otherwise 64 bf16.
static int prepare_gemm(const void* A, long long a_ld, long long a_seg_rows, int M_seg, int n_seg, int K,
                        const mmdit_linear_t& lin, int N, GemmParams p, uint16_t* wdeq, cudaStream_t st,
                        GemmProblem& out) {
  const bool f8 = p.ascale != nullptr;
  const int kb = f8 ? 128 : kBK, eb = f8 ? 1 : 2;  // K elements per stage, bytes per element
  if (K % kb || N % 32 || M_seg < 1 || n_seg < 1) return MMDIT_ERR_SHAPE;
  if (p.mode == GM_SWIGLU && N % kBN) return MMDIT_ERR_SHAPE;  // whole 128-row gate / up halves
  if (!al16(A) || (a_ld * eb) % 16) return MMDIT_ERR_ALIGN;
  const void* W = lin.w;
  p.wscale = nullptr;
  if (f8) {
    if (!lin.scale) return MMDIT_ERR_ARG;
    p.wscale = lin.scale;
    p.ascale_seg_rows = a_seg_rows;
  } else if (lin.scale) {
    if (!wdeq) return MMDIT_ERR_WORKSPACE;
    MMDIT_CUDA(launch_dequant_i8(static_cast<const int8_t*>(lin.w), wdeq, (long long)N * K, st));
    W = wdeq;
    p.wscale = lin.scale;
  }
  p.bias = lin.b;
  const CUtensorMapDataType dt = f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!make_tmap_3d(&out.ta, A, dt, eb, (uint64_t)K, (uint64_t)M_seg, (uint64_t)n_seg, (uint64_t)a_ld * eb,
                    (uint64_t)a_seg_rows * a_ld * eb, kb, kBM, true))
    return MMDIT_ERR_ALIGN;
  // W is loaded in 128-row halves of the 256-row tile, one by each CTA of a cluster pair.
  if (!make_tmap_3d(&out.tb, W, dt, eb, (uint64_t)K, (uint64_t)N, 1, (uint64_t)K * eb, (uint64_t)N * K * eb, kb,
                    kBN / 2, true))
    return MMDIT_ERR_ALIGN;
  // GM_RESID: the epilogue adds gate * value into the fp32 residual with TMA
  // reduce-adds of 32-row x 32-column boxes (rows at or beyond M_seg clipped).
  std::memset(&out.tr, 0, sizeof(out.tr));
  if (p.mode == GM_RESID &&
      (!p.resid || !make_tmap_3d(&out.tr, p.resid, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)N, (uint64_t)M_seg,
                                 (uint64_t)n_seg, (uint64_t)p.resid_ld * 4, (uint64_t)p.resid_seg_rows * p.resid_ld * 4,
                                 32, 32, true)))
    return MMDIT_ERR_ALIGN;
  out.f8 = f8;
  p.M_seg = M_seg;
  p.n_seg = n_seg;
  p.N = N;
  p.K = K;
  p.tiles_m = (M_seg + kBM - 1) / kBM;
  // SwiGLU: N = 2 x output width; an N tile pairs 128 gate rows with the 128 matching up rows
  p.swiglu_up = p.mode == GM_SWIGLU ? N / 2 : 0;
  p.tiles_n = p.mode == GM_SWIGLU ? (N / 2) / (kBN / 2) : (N + kBN - 1) / kBN;
  // Work units are pairs of vertically adjacent M tiles (one per CTA of a
  // cluster) at one N tile.
  const int pairs_m = (p.tiles_m * n_seg + 1) / 2;
  p.num_tiles = pairs_m * p.tiles_n;
  // Raster: when the whole A operand fits comfortably in L2, sweep all M
  // tiles for each N tile (A stays resident, W streams once); otherwise
  // groups of 8 pairs (16 M tiles) bound the A footprint of a wave.
  const double a_bytes = (double)n_seg * M_seg * K * eb;
  p.group_m = a_bytes <= 48.0 * 1024 * 1024 ? pairs_m : 8;
  p.status = device_status_ptr();
  out.p = p;
  return MMDIT_OK;
}

// One persistent launch over the tiles of one or two problems.
static int launch_problems(const GemmProblem* a, const GemmProblem* b, cudaStream_t st) {
  GemmGroup g;
  std::memset(&g, 0, sizeof(g));
  g.tmA[0] = a->ta;
  g.tmB[0] = a->tb;
  g.tmR[0] = a->tr;
  g.p[0] = a->p;
  g.n_prob = 1;
  g.f8 = a->f8 ? 1 : 0;
  if (b && b->f8 != a->f8) return MMDIT_ERR_ARG;
  g.tiles0 = a->p.num_tiles;
  g.total_tiles = g.tiles0;
  if (b) {
    g.tmA[1] = b->ta;
    g.tmB[1] = b->tb;
    g.tmR[1] = b->tr;
    g.p[1] = b->p;
    g.n_prob = 2;
    g.total_tiles += b->p.num_tiles;
  }
  return cuda_status(launch_gemm(g, st));
}

static int run_gemm(const void* A, long long a_ld, long long a_seg_rows, int M_seg, int n_seg, int K,
                    const mmdit_linear_t& lin, int N, GemmParams p, uint16_t* wdeq, cudaStream_t st) {
  GemmProblem pr;
  MMDIT_TRY(prepare_gemm(A, a_ld, a_seg_rows, M_seg, n_seg, K, lin, N, p, wdeq, st, pr));
  return launch_problems(&pr, nullptr, st);
}

static GemmParams gemm_params(int mode) {
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.mode = mode;
  p.gelu_from = 1 << 30;
  return p;
}

// ----------------------------------------------------------------- attention
int run_attention_prepared(int B, int L, int H, int d_head, int Lpad, const uint16_t* qk, const uint16_t* vT,
                           uint16_t* out, long long out_ld, int* merge_cnt, float* merge_part, cudaStream_t st,
                           bool merge_cnt_zero) {
  CUtensorMap tq, tv;
  const int D = H * d_head;
  const uint64_t D2 = 2ull * D;
  if (!make_tmap_3d(&tq, qk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D2, (uint64_t)L, (uint64_t)B, D2 * 2, D2 * 2 * L,
                    64, kAttnBM, true))
    return MMDIT_ERR_ALIGN;
  // The key extent of V^T is L (not Lpad): keys at or beyond L read as zeros.
  if (!make_tmap_3d(&tv, vT, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)L, (uint64_t)D, (uint64_t)B,
                    (uint64_t)Lpad * 2, (uint64_t)Lpad * 2 * D, 64, (uint32_t)d_head, true))
    return MMDIT_ERR_ALIGN;
  // Output rows of D columns at a pitch of out_ld elements, written by 32-row
  // TMA tile stores; rows at or beyond L are clipped.
  CUtensorMap to;
  if (!make_tmap_3d(&to, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)D, (uint64_t)L, (uint64_t)B,
                    (uint64_t)out_ld * 2, (uint64_t)out_ld * 2 * L, 64, 32, true))
    return MMDIT_ERR_ALIGN;
  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  p.L = L;
  p.H = H;
  p.B = B;
  p.n_q_tiles = (L + kAttnBM - 1) / kAttnBM;
  p.n_kv_tiles = (L + kAttnBN - 1) / kAttnBN;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d_head));
  p.status = device_status_ptr();
  p.cnt = merge_cnt;
  p.part = merge_part;
  p.cnt_zero = merge_cnt_zero ? 1 : 0;
  return cuda_status(launch_attention(tq, tv, to, p, d_head, st));
}

// Merge area of the persistent attention's split tail units (counters, then
// partial-result slots), carved from a workspace.
struct AttnMerge {
  int* cnt;
  float* part;
  size_t cnt_bytes;
  bool zeroed;  // cnt cleared by the caller (then every launch leaves it zero)
};
static void take_attn_merge(const Dims& d, Carve& c, AttnMerge& m) {
  const long long units = attn_units(d.B, d.L, d.H);
  m.cnt_bytes = attn_merge_ctas(units) * 8 * sizeof(int);
  m.cnt = c.take<int>(attn_merge_ctas(units) * 8);
  m.part = c.take<float>(attn_merge_floats(d.d, units));
  m.zeroed = false;
}
// One clear of the merge counters before a loop of blocks that share them.
static int clear_attn_merge(AttnMerge& m, cudaStream_t st) {
  const int rc = cuda_status(cudaMemsetAsync(m.cnt, 0, m.cnt_bytes, st));
  m.zeroed = rc == MMDIT_OK;
  return rc;
}

static int run_attention(const Dims& d, const uint16_t* qk, const uint16_t* vT, uint16_t* out, long long out_ld,
                         const AttnMerge& m, cudaStream_t st) {
  return run_attention_prepared(d.B, d.L, d.H, d.d, d.Lpad, qk, vT, out, out_ld, m.cnt, m.part, st, m.zeroed);
}

// ----------------------------------------------------------------- workspace layouts
struct DoubleWS {
  float* mod;
  uint16_t *y, *qk, *vT, *O, *h, *wdeq[2];
  uint8_t* a8;  // FP8: e4m3 copy of the current GEMM input (all rows), and its row scales
  float* as;
  AttnMerge am;
};
// y and h hold both streams at once (text rows first), so that each linear
// of the two streams runs as one grouped launch; int8 weights need one
// widening buffer per stream.
static void layout_double(const Dims& d, bool i8, bool need_mod, Carve& c, DoubleWS& w) {
  w.mod = need_mod ? c.take<float>((size_t)2 * d.B * 6 * d.D) : nullptr;
  w.y = c.take<uint16_t>((size_t)d.B * d.L * d.D);
  w.qk = c.take<uint16_t>((size_t)d.B * d.L * 2 * d.D);
  w.vT = c.take<uint16_t>((size_t)d.B * d.D * d.Lpad);
  w.O = c.take<uint16_t>((size_t)d.B * d.L * d.D);
  w.h = c.take<uint16_t>((size_t)d.B * d.L * d.Dm);
  const size_t wmlp = (size_t)(d.swiglu ? 2 : 1) * d.Dm;
  const size_t wmax = ((size_t)3 * d.D > wmlp ? (size_t)3 * d.D : wmlp) * d.D;
  w.wdeq[0] = i8 ? c.take<uint16_t>(wmax) : nullptr;
  w.wdeq[1] = i8 ? c.take<uint16_t>(wmax) : nullptr;
  w.a8 = d.f8 ? c.take<uint8_t>((size_t)d.B * d.L * (d.D > d.Dm ? d.D : d.Dm)) : nullptr;
  w.as = d.f8 ? c.take<float>((size_t)d.B * d.L) : nullptr;
  take_attn_merge(d, c, w.am);
}

struct SingleWS {
  float* mod;
  uint16_t *y, *qk, *vT, *cat, *wdeq;
  uint8_t* a8;
  float* as;
  AttnMerge am;
};
static void layout_single(const Dims& d, bool i8, bool need_mod, Carve& c, SingleWS& w) {
  w.mod = need_mod ? c.take<float>((size_t)d.B * 3 * d.D) : nullptr;
  w.y = c.take<uint16_t>((size_t)d.B * d.L * d.D);
  w.qk = c.take<uint16_t>((size_t)d.B * d.L * 2 * d.D);
  w.vT = c.take<uint16_t>((size_t)d.B * d.D * d.Lpad);
  w.cat = c.take<uint16_t>((size_t)d.B * d.L * (d.D + d.Dm));
  w.wdeq = i8 ? c.take<uint16_t>(((size_t)3 * d.D + (size_t)(d.swiglu ? 2 : 1) * d.Dm) * d.D) : nullptr;
  w.a8 = d.f8 ? c.take<uint8_t>((size_t)d.B * d.L * (d.D + d.Dm)) : nullptr;
  w.as = d.f8 ? c.take<float>((size_t)d.B * d.L) : nullptr;
  take_attn_merge(d, c, w.am);
}

struct StepWS {
  float *vec, *temb, *mods, *x, *v, *cs, *sn;
  uint16_t* xlat;
  uint8_t* block;
  size_t block_bytes;
};
static size_t mods_floats(const Dims& d, int n_double, int n_single) {
  return (size_t)n_double * 2 * d.B * 6 * d.D + (size_t)n_single * d.B * 3 * d.D + (size_t)d.B * 2 * d.D;
}
static void layout_step(const Dims& d, const mmdit_shape_t& s, int n_double, int n_single, Carve& c, StepWS& w) {
  const bool i8 = s.w_dtype == MMDIT_I8W;
  w.vec = c.take<float>((size_t)d.B * d.D);
  w.temb = c.take<float>((size_t)d.B * (s.t_dim + d.D));
  w.mods = c.take<float>(mods_floats(d, n_double, n_single));
  w.x = c.take<float>((size_t)d.B * d.L * d.D);
  w.v = c.take<float>((size_t)d.B * d.Lg * s.C_lat);
  w.xlat = c.take<uint16_t>((size_t)d.B * d.Li * s.C_lat);  // bf16 target latents, then reference latents
  w.cs = c.take<float>((size_t)d.L * (d.d / 2));
  w.sn = c.take<float>((size_t)d.L * (d.d / 2));
  Carve c1{nullptr, 0}, c2{nullptr, 0};
  DoubleWS dw;
  SingleWS sw;
  layout_double(d, i8, false, c1, dw);
  layout_single(d, i8, false, c2, sw);
  w.block_bytes = (c1.off > c2.off ? c1.off : c2.off) + 256;
  w.block = c.take<uint8_t>(w.block_bytes);
}

// ----------------------------------------------------------------- blocks
static int double_block_impl(const mmdit_shape_t& s, const Dims& d, const mmdit_double_w_t& w, const float* vec,
                             const float* mod_pre, float* x_txt, long long xt_seg_rows, float* x_img,
                             long long xi_seg_rows, const float* cs, const float* sn, const DoubleWS& ws,
                             cudaStream_t st) {
  const int D = d.D;
  const float* mod = mod_pre;
  if (!mod) {
    for (int i = 0; i < 2; ++i)
      MMDIT_CUDA(launch_gemv(w.mod[i].w, w.mod[i].scale != nullptr, w.mod[i].scale, w.mod[i].b, vec, d.B, 6 * D, D,
                             1, ws.mod + (size_t)i * d.B * 6 * D, st));
    mod = ws.mod;
  }
  float* xs[2] = {x_txt, x_img};
  const long long xseg[2] = {xt_seg_rows, xi_seg_rows};
  const int Ls[2] = {d.Lt, d.Li};
  const int off[2] = {0, d.Lt};
  const int first = d.Lt > 0 ? 0 : 1;  // streams with tokens: [first, 2)
  auto modp = [&](int i) { return mod + (size_t)i * d.B * 6 * D; };
  auto yp = [&](int i) { return ws.y + (size_t)off[i] * d.B * D; };
  auto hp = [&](int i) { return ws.h + (size_t)off[i] * d.B * d.Dm; };
  // Runs one linear of both streams as one grouped launch (text tiles first).
  auto grouped = [&](const GemmProblem* pr) -> int {
    return launch_problems(&pr[first], first == 0 ? &pr[1] : nullptr, st);
  };
  // FP8: a linear reads the e4m3 copy of its bf16 input, made by one row
  // quantisation pass over all B L rows (K wide) into ws.a8 / ws.as; stream
  // i's A operand and row scales start at the same row offset.
  auto quant = [&](const uint16_t* src, int K) -> int {
    return cuda_status(launch_quantize_f8(src, true, (long long)d.B * d.L, K, K, ws.a8, K, ws.as, st));
  };
  auto a_op = [&](const uint16_t* src, long long row0, int K, GemmParams& p) -> const void* {
    if (!d.f8) return src + row0 * K;
    p.ascale = ws.as + row0;
    return ws.a8 + row0 * K;
  };
  // LN + modulate of both streams in one launch at modulation chunk c (shift c, scale c + 1); with FP8 it
  // writes the e4m3 rows and their scales straight into ws.a8 / ws.as (at each stream's row offset) instead
  // of bf16 rows
  auto ln_mod = [&](int c) -> int {
    LnJob jobs[2];
    int n = 0;
    for (int i = first; i < 2; ++i) {
      const long long r0 = (long long)off[i] * d.B;
      jobs[n++] = LnJob{xs[i], xseg[i], Ls[i], d.B, modp(i) + (size_t)c * D, modp(i) + (size_t)(c + 1) * D, 6 * D,
                        d.f8 ? nullptr : yp(i), d.f8 ? ws.a8 + r0 * D : nullptr, d.f8 ? ws.as + r0 : nullptr};
    }
    return cuda_status(launch_ln_modulate_jobs(jobs, n, D, s.eps_ln, st));
  };
  GemmProblem pr[2];
  // LN + modulate, then the fused QKV / RMSNorm / RoPE GEMM
  MMDIT_TRY(ln_mod(0));
  for (int i = first; i < 2; ++i) {
    GemmParams p = gemm_params(GM_QKV);
    p.out_seg_rows = d.L;
    p.out_row_off = off[i];
    p.qkv_D = D;
    p.d_head = d.d;
    p.gq = w.q_norm[i];
    p.gk = w.k_norm[i];
    p.eps = s.eps_rms;
    p.rope_cos = cs;
    p.rope_sin = sn;
    p.qk = ws.qk;
    p.qk_ld = 2 * D;
    p.vT = ws.vT;
    p.vT_ld = d.Lpad;
    const void* A = a_op(ws.y, (long long)off[i] * d.B, D, p);
    MMDIT_TRY(prepare_gemm(A, D, Ls[i], Ls[i], d.B, D, w.qkv[i], 3 * D, p, ws.wdeq[i], st, pr[i]));
  }
  MMDIT_TRY(grouped(pr));
  MMDIT_TRY(run_attention(d, ws.qk, ws.vT, ws.O, D, ws.am, st));
  if (d.f8) MMDIT_TRY(quant(ws.O, D));
  // x += gate1 * (o Wp^T + bp)
  for (int i = first; i < 2; ++i) {
    GemmParams p = gemm_params(GM_RESID);
    p.resid = xs[i];
    p.resid_ld = D;
    p.resid_seg_rows = xseg[i];
    p.gate = modp(i) + 2 * D;
    p.gate_seg_stride = 6 * D;
    const void* A = a_op(ws.O, off[i], D, p);
    MMDIT_TRY(prepare_gemm(A, D, d.L, Ls[i], d.B, D, w.proj[i], D, p, ws.wdeq[i], st, pr[i]));
  }
  MMDIT_TRY(grouped(pr));
  // y2 = LN(x)(1 + scale2) + shift2; h = GELU(y2 W1^T + b1)
  MMDIT_TRY(ln_mod(3));
  for (int i = first; i < 2; ++i) {
    GemmParams p = gemm_params(d.swiglu ? GM_SWIGLU : GM_STORE_BF16);
    p.gelu_from = 0;
    p.out = hp(i);
    p.out_ld = d.Dm;
    p.out_seg_rows = Ls[i];
    const void* A = a_op(ws.y, (long long)off[i] * d.B, D, p);
    MMDIT_TRY(prepare_gemm(A, D, Ls[i], Ls[i], d.B, D, w.mlp_in[i], d.swiglu ? 2 * d.Dm : d.Dm, p, ws.wdeq[i], st,
                           pr[i]));
  }
  MMDIT_TRY(grouped(pr));
  if (d.f8) MMDIT_TRY(quant(ws.h, d.Dm));
  // x += gate2 * (h W2^T + b2)
  for (int i = first; i < 2; ++i) {
    GemmParams p = gemm_params(GM_RESID);
    p.resid = xs[i];
    p.resid_ld = D;
    p.resid_seg_rows = xseg[i];
    p.gate = modp(i) + 5 * D;
    p.gate_seg_stride = 6 * D;
    const void* A = a_op(ws.h, (long long)off[i] * d.B, d.Dm, p);
    MMDIT_TRY(prepare_gemm(A, d.Dm, Ls[i], Ls[i], d.B, d.Dm, w.mlp_out[i], D, p, ws.wdeq[i], st, pr[i]));
  }
  MMDIT_TRY(grouped(pr));
  return MMDIT_OK;
}

static int single_block_impl(const mmdit_shape_t& s, const Dims& d, const mmdit_single_w_t& w, const float* vec,
                             const float* mod_pre, float* x, const float* cs, const float* sn, const SingleWS& ws,
                             cudaStream_t st) {
  const int D = d.D;
  const float* mod = mod_pre;
  if (!mod) {
    MMDIT_CUDA(launch_gemv(w.mod.w, w.mod.scale != nullptr, w.mod.scale, w.mod.b, vec, d.B, 3 * D, D, 1, ws.mod, st));
    mod = ws.mod;
  }
  // FP8: lin1 reads the e4m3 rows of y (written by LN + modulate itself), lin2 those of [O | act(mlp)]
  MMDIT_CUDA(launch_ln_modulate(x, d.L, d.L, d.B, D, mod, mod + D, 3 * D, s.eps_ln, d.f8 ? nullptr : ws.y, st,
                                d.f8 ? ws.a8 : nullptr, d.f8 ? ws.as : nullptr));
  const long long cat_ld = D + d.Dm;
  const long long rows = (long long)d.B * d.L;
  const void* A1 = d.f8 ? static_cast<const void*>(ws.a8) : static_cast<const void*>(ws.y);
  GemmParams p = gemm_params(GM_QKV);
  p.ascale = d.f8 ? ws.as : nullptr;
  p.out_seg_rows = d.L;
  p.out_row_off = 0;
  p.qkv_D = D;
  p.d_head = d.d;
  p.gq = w.q_norm;
  p.gk = w.k_norm;
  p.eps = s.eps_rms;
  p.rope_cos = cs;
  p.rope_sin = sn;
  p.qk = ws.qk;
  p.qk_ld = 2 * D;
  p.vT = ws.vT;
  p.vT_ld = d.Lpad;
  p.aux = ws.cat;
  p.aux_ld = cat_ld;
  p.aux_col_off = D;
  if (!d.swiglu) {
    MMDIT_TRY(run_gemm(A1, D, d.L, d.L, d.B, D, w.lin1, 3 * D + d.Dm, p, ws.wdeq, st));
  } else {
    // lin1 rows [q; k; v] (QKV epilogue) and [gate; up] (SwiGLU into the columns
    // [D, D + Dm) of cat) as the two problems of one launch
    const bool i8 = w.lin1.scale != nullptr;
    const size_t wb = i8 ? 1 : 2;
    mmdit_linear_t mlp = w.lin1;
    mlp.w = static_cast<const uint8_t*>(w.lin1.w) + (size_t)3 * D * D * wb;
    if (w.lin1.b) mlp.b = static_cast<const float*>(w.lin1.b) + 3 * D;
    if (w.lin1.scale) mlp.scale = w.lin1.scale + 3 * D;
    GemmProblem pr[2];
    MMDIT_TRY(prepare_gemm(A1, D, d.L, d.L, d.B, D, w.lin1, 3 * D, p, ws.wdeq, st, pr[0]));
    GemmParams ps = gemm_params(GM_SWIGLU);
    ps.ascale = p.ascale;
    ps.out = ws.cat + D;
    ps.out_ld = cat_ld;
    ps.out_seg_rows = d.L;
    MMDIT_TRY(prepare_gemm(A1, D, d.L, d.L, d.B, D, mlp, 2 * d.Dm, ps, ws.wdeq ? ws.wdeq + (size_t)3 * D * D : nullptr,
                           st, pr[1]));
    MMDIT_TRY(launch_problems(&pr[0], &pr[1], st));
  }
  MMDIT_TRY(run_attention(d, ws.qk, ws.vT, ws.cat, cat_ld, ws.am, st));
  if (d.f8) MMDIT_CUDA(launch_quantize_f8(ws.cat, true, rows, (int)cat_ld, cat_ld, ws.a8, cat_ld, ws.as, st));
  GemmParams p2 = gemm_params(GM_RESID);
  p2.ascale = d.f8 ? ws.as : nullptr;
  p2.resid = x;
  p2.resid_ld = D;
  p2.resid_seg_rows = d.L;
  p2.gate = mod + 2 * D;
  p2.gate_seg_stride = 3 * D;
  MMDIT_TRY(run_gemm(d.f8 ? static_cast<const void*>(ws.a8) : static_cast<const void*>(ws.cat), cat_ld, d.L, d.L, d.B,
                     (int)cat_ld, w.lin2, D, p2, ws.wdeq, st));
  return MMDIT_OK;
}

// Which linears carry a per-channel scale: every linear for int8 weights;
// only the block GEMM linears for FP8 (modulation stays bf16).
static bool scaled_gemv(int w_dtype) { return w_dtype == MMDIT_I8W; }
static bool scaled_gemm(int w_dtype) { return w_dtype == MMDIT_I8W || w_dtype == MMDIT_F8W; }

static bool double_w_ok(const mmdit_double_w_t* w, int w_dtype) {
  if (!w) return false;
  const bool qv = scaled_gemv(w_dtype), qg = scaled_gemm(w_dtype);
  for (int i = 0; i < 2; ++i) {
    if (!lin_ok(w->mod[i], qv) || !lin_ok(w->qkv[i], qg) || !lin_ok(w->proj[i], qg) || !lin_ok(w->mlp_in[i], qg) ||
        !lin_ok(w->mlp_out[i], qg))
      return false;
    if (!w->q_norm[i] || !w->k_norm[i] || !al16(w->q_norm[i]) || !al16(w->k_norm[i])) return false;
  }
  return true;
}

static bool single_w_ok(const mmdit_single_w_t* w, int w_dtype) {
  if (!w) return false;
  const bool qv = scaled_gemv(w_dtype), qg = scaled_gemm(w_dtype);
  if (!lin_ok(w->mod, qv) || !lin_ok(w->lin1, qg) || !lin_ok(w->lin2, qg)) return false;
  return w->q_norm && w->k_norm && al16(w->q_norm) && al16(w->k_norm);
}

static int step_w_check(const mmdit_shape_t& shape, const mmdit_step_w_t& w) {
  if (w.n_double < 0 || w.n_single < 0 || (w.n_double && !w.doubles) || (w.n_single && !w.singles))
    return MMDIT_ERR_ARG;
  const bool i8 = shape.w_dtype == MMDIT_I8W;
  if (!lin_ok(w.time1, i8) || !lin_ok(w.time2, i8) || !lin_ok(w.img_in, i8) || !lin_ok(w.final_mod, i8) ||
      !lin_ok(w.final, i8))
    return MMDIT_ERR_ARG;
  for (int i = 0; i < w.n_double; ++i)
    if (!double_w_ok(&w.doubles[i], shape.w_dtype)) return MMDIT_ERR_ARG;
  for (int i = 0; i < w.n_single; ++i)
    if (!single_w_ok(&w.singles[i], shape.w_dtype)) return MMDIT_ERR_ARG;
  return MMDIT_OK;
}

// ----------------------------------------------------------------- step
// One denoising step on the laid-out step workspace sw.  vec_add (or null)
// is added to the timestep embedding.  With sig_tab / sig_idx set, sigma and
// sigma_next are read on the device as sig_tab[k], sig_tab[k + 1] with
// k = *sig_idx (the host values are ignored), so one captured step replays
// for every step of a schedule.
// The modulation linears of every block and of the final layer, in the
// order of their vectors in a step's modulation buffer `base`: a double
// block's two streams ([B][6D] each), a single block's [B][3D], the final
// layer's [B][2D].  Output row b of a job goes to out + b * ldo (ldo 0: N).
static std::vector<GemvJob> mod_jobs(const Dims& d, const mmdit_step_w_t& w, float* base, long long ldo) {
  const int D = d.D;
  std::vector<GemvJob> jobs;
  float* mp = base;
  const size_t rows = ldo ? 1 : (size_t)d.B;  // with a row stride, one row's outputs per job slot
  for (int i = 0; i < w.n_double; ++i)
    for (int s = 0; s < 2; ++s) {
      const mmdit_linear_t& l = w.doubles[i].mod[s];
      jobs.push_back(GemvJob{l.w, l.scale, l.b, mp, 6 * D, ldo});
      mp += rows * 6 * D;
    }
  for (int i = 0; i < w.n_single; ++i) {
    const mmdit_linear_t& l = w.singles[i].mod;
    jobs.push_back(GemvJob{l.w, l.scale, l.b, mp, 3 * D, ldo});
    mp += rows * 3 * D;
  }
  jobs.push_back(GemvJob{w.final_mod.w, w.final_mod.scale, w.final_mod.b, mp, 2 * D, ldo});
  return jobs;
}

// mods_all: the modulation buffers of every step of a sampling run, computed
// beforehand (step k's at mods_all + k * mods_floats); step_impl then copies
// step k's (k = *sig_idx on the device, or step_k) instead of evaluating the
// timestep embedding and the modulation linears.
static int step_impl(const mmdit_shape_t& shape, const Dims& d, const mmdit_step_w_t& w, float* x_lat,
                     const float* x_ref, const float* x_txt_in, double sigma, double sigma_next, float* v_out,
                     const float* vec_add,
                     const double* sig_tab, const int* sig_idx, bool build_rope, const StepWS& sw, cudaStream_t st,
                     const float* mods_all = nullptr, int step_k = 0) {
  const bool i8 = shape.w_dtype == MMDIT_I8W;
  const int D = d.D, C = shape.C_lat;
  if (build_rope)
    MMDIT_CUDA(launch_rope_build(d.Lt, shape.grid_w, d.Lg, shape.ref_w, d.L, shape.rope_axes, shape.rope_theta,
                                 nullptr, sw.cs, sw.sn, st));
  const long long mods_n = (long long)mods_floats(d, w.n_double, w.n_single);
  if (mods_all) {
    MMDIT_CUDA(launch_select_step(mods_all, mods_n, mods_n, sig_idx, step_k, sw.mods, st));
  } else {
    // timestep embedding: vec = time2 SiLU(time1 sinusoid(1000 sigma))
    MMDIT_CUDA(launch_sinusoid(1000.0 * sigma, d.B, shape.t_dim, sw.temb, st, sig_tab, sig_idx, 1000.0));
    float* th = sw.temb + (size_t)d.B * shape.t_dim;
    MMDIT_CUDA(launch_gemv(w.time1.w, w.time1.scale != nullptr, w.time1.scale, w.time1.b, sw.temb, d.B, D,
                           shape.t_dim, 0, th, st));
    MMDIT_CUDA(launch_gemv(w.time2.w, w.time2.scale != nullptr, w.time2.scale, w.time2.b, th, d.B, D, D, 1,
                           sw.vec, st));
    if (vec_add) MMDIT_CUDA(launch_add(sw.vec, vec_add, (long long)d.B * D, st));
    // modulation vectors of every block and of the final layer (they depend on vec only): one batched launch
    const std::vector<GemvJob> jobs = mod_jobs(d, w, sw.mods, 0);
    MMDIT_CUDA(launch_gemv_batched(jobs.data(), (int)jobs.size(), i8, sw.vec, d.B, D, 1, st));
  }
  float* const mod_final = sw.mods + mods_n - (size_t)d.B * 2 * D;
  // residual stream x = [text; image] per sample: text copied in, image from img_in
  if (d.Lt > 0)
    MMDIT_CUDA(cudaMemcpy2DAsync(sw.x, (size_t)d.L * D * 4, x_txt_in, (size_t)d.Lt * D * 4, (size_t)d.Lt * D * 4, d.B,
                                 cudaMemcpyDeviceToDevice, st));
  // img_in: the target latents into image rows [0, Lg) of each sample, the reference latents (if any) into
  // rows [Lg, Li), as the two problems of one launch
  uint16_t* xref16 = sw.xlat + (size_t)d.B * d.Lg * C;
  MMDIT_CUDA(launch_cast_bf16(x_lat, sw.xlat, (long long)d.B * d.Lg * C, st));
  if (d.Lr > 0) MMDIT_CUDA(launch_cast_bf16(x_ref, xref16, (long long)d.B * d.Lr * C, st));
  {
    GemmParams p = gemm_params(GM_STORE_F32);
    p.out = sw.x;
    p.out_ld = D;
    p.out_seg_rows = d.L;
    p.out_row_off = d.Lt;
    Carve bc{sw.block, 0};
    uint16_t* wdeq = i8 ? bc.take<uint16_t>((size_t)D * C) : nullptr;
    GemmProblem pr[2];
    MMDIT_TRY(prepare_gemm(sw.xlat, C, d.Lg, d.Lg, d.B, C, w.img_in, D, p, wdeq, st, pr[0]));
    if (d.Lr > 0) {
      p.out_row_off = d.Lt + d.Lg;
      // int8 weights were widened into wdeq by the first problem's preparation: the second reads that copy,
      // with the same per-channel scale in its epilogue
      const mmdit_linear_t lin = wdeq ? mmdit_linear_t{wdeq, w.img_in.b, nullptr} : w.img_in;
      MMDIT_TRY(prepare_gemm(xref16, C, d.Lr, d.Lr, d.B, C, lin, D, p, nullptr, st, pr[1]));
      if (wdeq) pr[1].p.wscale = w.img_in.scale;
    }
    MMDIT_TRY(launch_problems(&pr[0], d.Lr > 0 ? &pr[1] : nullptr, st));
  }
  // blocks
  float* mp = sw.mods;
  {
    Carve bc{sw.block, 0};
    DoubleWS dw;
    layout_double(d, i8, false, bc, dw);
    if (w.n_double > 0) MMDIT_TRY(clear_attn_merge(dw.am, st));
    for (int i = 0; i < w.n_double; ++i) {
      MMDIT_TRY(double_block_impl(shape, d, w.doubles[i], nullptr, mp, sw.x, d.L, sw.x + (size_t)d.Lt * D, d.L,
                                  sw.cs, sw.sn, dw, st));
      mp += (size_t)2 * d.B * 6 * D;
    }
  }
  {
    Carve bc{sw.block, 0};
    SingleWS ssw;
    layout_single(d, i8, false, bc, ssw);
    if (w.n_single > 0) MMDIT_TRY(clear_attn_merge(ssw.am, st));
    for (int i = 0; i < w.n_single; ++i) {
      MMDIT_TRY(single_block_impl(shape, d, w.singles[i], nullptr, mp, sw.x, sw.cs, sw.sn, ssw, st));
      mp += (size_t)d.B * 3 * D;
    }
  }
  // final layer on the image tokens and the Euler update
  {
    Carve bc{sw.block, 0};
    uint16_t* y = bc.take<uint16_t>((size_t)d.B * d.Lg * D);
    uint16_t* wdeq = i8 ? bc.take<uint16_t>((size_t)D * C) : nullptr;
    MMDIT_CUDA(launch_ln_modulate(sw.x + (size_t)d.Lt * D, d.L, d.Lg, d.B, D, mod_final, mod_final + D, 2 * D,
                                  shape.eps_ln, y, st));
    GemmParams p = gemm_params(GM_STORE_F32);
    float* v = v_out ? v_out : sw.v;
    p.out = v;
    p.out_ld = C;
    p.out_seg_rows = d.Lg;
    MMDIT_TRY(run_gemm(y, D, d.Lg, d.Lg, d.B, D, w.final, C, p, wdeq, st));
    MMDIT_CUDA(launch_euler(x_lat, v, false, (float)(sigma_next - sigma), (long long)d.B * d.Lg * C, st, sig_tab,
                            sig_idx));
  }
  return MMDIT_OK;
}


}  // namespace mmdit

using namespace mmdit;

// =================================================================== exports
extern "C" {

const char* mmdit_status_string(int status) {
  switch (status) {
    case MMDIT_OK: return "ok";
    case MMDIT_ERR_ARG: return "invalid argument (null pointer or bad enum)";
    case MMDIT_ERR_SHAPE: return "shape outside the supported limits";
    case MMDIT_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
    case MMDIT_ERR_WORKSPACE: return "workspace too small";
    case MMDIT_ERR_CUDA: return "CUDA runtime error";
    case MMDIT_ERR_TIMEOUT: return "a kernel abandoned a bounded wait";
    case MMDIT_ERR_UNSUPPORTED: return "device is not sm_103 or a driver entry point is missing";
    default: return "unknown status";
  }
}

int mmdit_sync_status(void* stream) {
  if (cudaStreamSynchronize(S(stream)) != cudaSuccess) return MMDIT_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(v)) != cudaSuccess) return MMDIT_ERR_CUDA;
  if (v) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess) return MMDIT_ERR_CUDA;
    return MMDIT_ERR_TIMEOUT;
  }
  return MMDIT_OK;
}

long long mmdit_launch_count(void) { return g_launches.load(); }

const char* mmdit_kernel_name(int kernel_id) {
  static const char* names[KID_COUNT] = {"gemm_bf16_tc", "attn_fwd",   "ln_modulate", "gemv",      "sinusoid",
                                         "rope_build",   "rope_apply", "euler",       "quantize_w8", "dequant_i8",
                                         "cast_bf16",    "attn_prep",  "wait_selftest", "add_f32",
                                         "step_counter", "quantize_f8", "heads_pack",   "heads_unpack",
                                         "vT_transpose", "select_step"};
  return (kernel_id >= 0 && kernel_id < KID_COUNT) ? names[kernel_id] : "unknown";
}

int mmdit_trace_begin(int capacity) {
  if (capacity < 1) return MMDIT_ERR_ARG;
  trace_free();
  g_trace.ev = new cudaEvent_t[2 * (size_t)capacity];
  g_trace.ids = new int[capacity];
  for (int i = 0; i < 2 * capacity; ++i) {
    if (cudaEventCreate(&g_trace.ev[i]) != cudaSuccess) {
      g_trace.cap = i / 2;
      trace_free();
      return MMDIT_ERR_CUDA;
    }
    g_trace.cap = (i + 1) / 2;
  }
  g_trace.cap = capacity;
  g_trace.n = 0;
  g_trace.on = true;
  return MMDIT_OK;
}

int mmdit_trace_end(int* count) {
  g_trace.on = false;
  if (count) *count = g_trace.n;
  return MMDIT_OK;
}

int mmdit_trace_read(int* kernel_ids, float* ms, int capacity, int* count) {
  if (!kernel_ids || !ms || !count || capacity < 0) return MMDIT_ERR_ARG;
  const int n = g_trace.n < capacity ? g_trace.n : capacity;
  for (int i = 0; i < n; ++i) {
    if (cudaEventSynchronize(g_trace.ev[2 * i + 1]) != cudaSuccess) return MMDIT_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, g_trace.ev[2 * i], g_trace.ev[2 * i + 1]) != cudaSuccess) return MMDIT_ERR_CUDA;
    kernel_ids[i] = g_trace.ids[i];
    ms[i] = t;
  }
  *count = n;
  return MMDIT_OK;
}

int mmdit_workspace_size(const mmdit_shape_t* shape, int op, size_t* bytes) {
  if (!bytes) return MMDIT_ERR_ARG;
  Dims d;
  MMDIT_TRY(check_shape(shape, &d));
  const bool i8 = shape->w_dtype == MMDIT_I8W;
  Carve c{nullptr, 0};
  switch (op) {
    case MMDIT_OP_DOUBLE: {
      DoubleWS w;
      layout_double(d, i8, true, c, w);
      break;
    }
    case MMDIT_OP_SINGLE: {
      SingleWS w;
      layout_single(d, i8, true, c, w);
      break;
    }
    case MMDIT_OP_ATTENTION: {
      c.take<uint16_t>((size_t)d.B * d.L * 2 * d.D);
      c.take<uint16_t>((size_t)d.B * d.D * d.Lpad);
      AttnMerge m;
      take_attn_merge(d, c, m);
      break;
    }
    default:
      return MMDIT_ERR_ARG;
  }
  *bytes = c.off + 256;
  return MMDIT_OK;
}

int mmdit_step_workspace_size(const mmdit_shape_t* shape, int n_double, int n_single, size_t* bytes) {
  if (!bytes || n_double < 0 || n_single < 0) return MMDIT_ERR_ARG;
  Dims d;
  MMDIT_TRY(check_shape(shape, &d));
  if (shape->C_lat <= 0 || shape->C_lat % 64 || shape->t_dim <= 0 || shape->t_dim % 16) return MMDIT_ERR_SHAPE;
  Carve c{nullptr, 0};
  StepWS w;
  layout_step(d, *shape, n_double, n_single, c, w);
  *bytes = c.off + 256;
  return MMDIT_OK;
}

int mmdit_rope2d_build(const mmdit_shape_t* shape, int32_t* ids, float* cos_, float* sin_, void* stream) {
  Dims d;
  MMDIT_TRY(check_shape(shape, &d));
  if (!cos_ || !sin_) return MMDIT_ERR_ARG;
  if (!al16(cos_) || !al16(sin_) || (ids && (reinterpret_cast<uintptr_t>(ids) & 3))) return MMDIT_ERR_ALIGN;
  MMDIT_TRY(check_device());
  return cuda_status(
      launch_rope_build(d.Lt, shape->grid_w, d.Lg, shape->ref_w, d.L, shape->rope_axes, shape->rope_theta, ids, cos_,
                        sin_, S(stream)));
}

int rope2d_apply(const mmdit_shape_t* shape, const float* cos_, const float* sin_, void* x, int row_stride,
                 void* stream) {
  Dims d;
  MMDIT_TRY(check_shape(shape, &d));
  if (!cos_ || !sin_ || !x) return MMDIT_ERR_ARG;
  if (row_stride < d.D || row_stride % 8) return MMDIT_ERR_SHAPE;
  if (!al16(cos_) || !al16(sin_) || !al16(x)) return MMDIT_ERR_ALIGN;
  MMDIT_TRY(check_device());
  return cuda_status(launch_rope_apply(static_cast<uint16_t*>(x), (long long)d.B * d.L, d.L, d.H, d.d, row_stride,
                                       cos_, sin_, S(stream)));
}

int joint_attention_fwd(const mmdit_shape_t* shape, const void* qkv, int qkv_row_stride, const float* const q_norm[2],
                        const float* const k_norm[2], const float* cos_, const float* sin_, void* out,
                        int out_row_stride, void* ws, size_t ws_bytes, void* stream) {
  Dims d;
  MMDIT_TRY(check_shape(shape, &d));
  if (!qkv || !out || !ws) return MMDIT_ERR_ARG;
  if ((cos_ == nullptr) != (sin_ == nullptr)) return MMDIT_ERR_ARG;
  if (qkv_row_stride < 3 * d.D || qkv_row_stride % 8 || out_row_stride < d.D || out_row_stride % 8)
    return MMDIT_ERR_SHAPE;
  if (!al16(qkv) || !al16(out) || !al16(ws)) return MMDIT_ERR_ALIGN;
  const float* gq0 = q_norm ? q_norm[0] : nullptr;
  const float* gq1 = q_norm ? q_norm[1] : nullptr;
  const float* gk0 = k_norm ? k_norm[0] : nullptr;
  const float* gk1 = k_norm ? k_norm[1] : nullptr;
  if (gq0 && (!gq1 || !gk0 || !gk1)) return MMDIT_ERR_ARG;
  size_t need = 0;
  MMDIT_TRY(mmdit_workspace_size(shape, MMDIT_OP_ATTENTION, &need));
  if (ws_bytes < need) return MMDIT_ERR_WORKSPACE;
  MMDIT_TRY(check_device());
  Carve c{static_cast<uint8_t*>(ws), 0};
  uint16_t* qk = c.take<uint16_t>((size_t)d.B * d.L * 2 * d.D);
  uint16_t* vT = c.take<uint16_t>((size_t)d.B * d.D * d.Lpad);
  AttnMerge am;
  take_attn_merge(d, c, am);
  MMDIT_CUDA(launch_attn_prep(static_cast<const uint16_t*>(qkv), qkv_row_stride, d.B, d.L, d.Lt, d.H, d.d, gq0, gq1,
                              gk0, gk1, shape->eps_rms, cos_, sin_, qk, vT, d.Lpad, S(stream)));
  return run_attention(d, qk, vT, static_cast<uint16_t*>(out), out_row_stride, am, S(stream));
}

int mmdit_double_block_fwd(const mmdit_shape_t* shape, const mmdit_double_w_t* w, const float* vec,
                           const float* mod_precomputed, float* x_txt, float* x_img, const float* cos_,
                           const float* sin_, void* ws, size_t ws_bytes, void* stream) {
  Dims d;
  MMDIT_TRY(check_shape(shape, &d));
  const bool i8 = shape->w_dtype == MMDIT_I8W;
  if (!double_w_ok(w, shape->w_dtype)) return MMDIT_ERR_ARG;
  if ((vec == nullptr) == (mod_precomputed == nullptr)) return MMDIT_ERR_ARG;
  if (!x_img || (d.Lt > 0 && !x_txt) || !cos_ || !sin_ || !ws) return MMDIT_ERR_ARG;
  if ((x_txt && !al16(x_txt)) || !al16(x_img) || !al16(cos_) || !al16(sin_) || !al16(ws) ||
      (vec && !al16(vec)) || (mod_precomputed && !al16(mod_precomputed)))
    return MMDIT_ERR_ALIGN;
  Carve c{static_cast<uint8_t*>(ws), 0};
  DoubleWS dw;
  {
    Carve q{nullptr, 0};
    layout_double(d, i8, vec != nullptr, q, dw);
    if (ws_bytes < q.off) return MMDIT_ERR_WORKSPACE;
  }
  MMDIT_TRY(check_device());
  layout_double(d, i8, vec != nullptr, c, dw);
  return double_block_impl(*shape, d, *w, vec, mod_precomputed, x_txt, d.Lt, x_img, d.Li, cos_, sin_, dw, S(stream));
}

int mmdit_single_block_fwd(const mmdit_shape_t* shape, const mmdit_single_w_t* w, const float* vec,
                           const float* mod_precomputed, float* x, const float* cos_, const float* sin_, void* ws,
                           size_t ws_bytes, void* stream) {
  Dims d;
  MMDIT_TRY(check_shape(shape, &d));
  const bool i8 = shape->w_dtype == MMDIT_I8W;
  if (!single_w_ok(w, shape->w_dtype)) return MMDIT_ERR_ARG;
  if ((vec == nullptr) == (mod_precomputed == nullptr)) return MMDIT_ERR_ARG;
  if (!x || !cos_ || !sin_ || !ws) return MMDIT_ERR_ARG;
  if (!al16(x) || !al16(cos_) || !al16(sin_) || !al16(ws) || (vec && !al16(vec)) ||
      (mod_precomputed && !al16(mod_precomputed)))
    return MMDIT_ERR_ALIGN;
  SingleWS sw;
  {
    Carve q{nullptr, 0};
    layout_single(d, i8, vec != nullptr, q, sw);
    if (ws_bytes < q.off) return MMDIT_ERR_WORKSPACE;
  }
  MMDIT_TRY(check_device());
  Carve c{static_cast<uint8_t*>(ws), 0};
  layout_single(d, i8, vec != nullptr, c, sw);
  return single_block_impl(*shape, d, *w, vec, mod_precomputed, x, cos_, sin_, sw, S(stream));
}

int mmdit_step_i2i_fwd(const mmdit_shape_t* shape, const mmdit_step_w_t* w, float* x_lat, const float* x_ref,
                       const float* x_txt_in, double sigma, double sigma_next, float* v_out, void* ws,
                       size_t ws_bytes, void* stream) {
  Dims d;
  MMDIT_TRY(check_shape(shape, &d));
  if (!w || !x_lat || (d.Lt > 0 && !x_txt_in) || !ws || (d.Lr > 0) != (x_ref != nullptr)) return MMDIT_ERR_ARG;
  MMDIT_TRY(step_w_check(*shape, *w));
  if (!al16(x_lat) || (x_ref && !al16(x_ref)) || (x_txt_in && !al16(x_txt_in)) || !al16(ws) ||
      (v_out && !al16(v_out)))
    return MMDIT_ERR_ALIGN;
  size_t need = 0;
  MMDIT_TRY(mmdit_step_workspace_size(shape, w->n_double, w->n_single, &need));
  if (ws_bytes < need) return MMDIT_ERR_WORKSPACE;
  MMDIT_TRY(check_device());
  Carve c{static_cast<uint8_t*>(ws), 0};
  StepWS sw;
  layout_step(d, *shape, w->n_double, w->n_single, c, sw);
  return step_impl(*shape, d, *w, x_lat, x_ref, x_txt_in, sigma, sigma_next, v_out, nullptr, nullptr, nullptr, true,
                   sw, S(stream));
}

int mmdit_step_fwd(const mmdit_shape_t* shape, const mmdit_step_w_t* w, float* x_lat, const float* x_txt_in,
                   double sigma, double sigma_next, float* v_out, void* ws, size_t ws_bytes, void* stream) {
  return mmdit_step_i2i_fwd(shape, w, x_lat, nullptr, x_txt_in, sigma, sigma_next, v_out, ws, ws_bytes, stream);
}

// Workspace of the sampling loop: the step's, then the conditioning.
struct SampleWS {
  float *x_txt, *vec_cond, *ctemb, *phid, *ptmp;
  double* sig;
  int* ctr;
  uint16_t* wdeq;
  float* vec_all;   // [B][n_steps][D]: every step's conditioning vector
  float* mods_all;  // [n_steps][mods_floats]: every step's modulation buffer
};
static void layout_sample(const Dims& d, const mmdit_shape_t& s, int n_double, int n_single, int C_txt, int n_steps,
                          Carve& c, SampleWS& w) {
  const bool i8 = s.w_dtype == MMDIT_I8W;
  w.vec_all = c.take<float>((size_t)d.B * n_steps * d.D);
  w.mods_all = c.take<float>((size_t)n_steps * mods_floats(d, n_double, n_single));
  w.x_txt = c.take<float>((size_t)d.B * d.Lt * d.D);
  w.vec_cond = c.take<float>((size_t)d.B * d.D);
  w.ctemb = c.take<float>((size_t)d.B * (s.t_dim + d.D));
  w.phid = c.take<float>((size_t)d.B * d.D);
  w.ptmp = c.take<float>((size_t)d.B * d.D);
  w.sig = c.take<double>((size_t)n_steps + 1);
  w.ctr = c.take<int>(4);
  w.wdeq = i8 ? c.take<uint16_t>((size_t)d.D * C_txt) : nullptr;
}

int mmdit_sample_workspace_size(const mmdit_shape_t* shape, int n_double, int n_single, int C_txt, int n_steps,
                                size_t* bytes) {
  if (!bytes || n_steps < 1 || C_txt <= 0) return MMDIT_ERR_ARG;
  size_t step = 0;
  MMDIT_TRY(mmdit_step_workspace_size(shape, n_double, n_single, &step));
  Dims d;
  MMDIT_TRY(check_shape(shape, &d));
  Carve c{nullptr, step};
  SampleWS w;
  layout_sample(d, *shape, n_double, n_single, C_txt, n_steps, c, w);
  *bytes = c.off + 256;
  return MMDIT_OK;
}

int mmdit_sample(const mmdit_shape_t* shape, const mmdit_step_w_t* w, const mmdit_cond_w_t* cond, float* x_lat,
                 const void* txt, const float* pooled, double guidance, const double* sigmas, int n_steps, int flags,
                 void* ws, size_t ws_bytes, void* stream) {
  Dims d;
  MMDIT_TRY(check_shape(shape, &d));
  if (!w || !cond || !x_lat || (d.Lt > 0 && !txt) || !pooled || !sigmas || !ws || n_steps < 1) return MMDIT_ERR_ARG;
  if (d.Lr > 0) return MMDIT_ERR_ARG;  // reference latents: step by step through mmdit_step_i2i_fwd
  if (flags & ~MMDIT_SAMPLE_GRAPH) return MMDIT_ERR_ARG;
  MMDIT_TRY(step_w_check(*shape, *w));
  const bool i8 = shape->w_dtype == MMDIT_I8W;
  if (!lin_ok(cond->txt_in, i8) || !lin_ok(cond->guid1, i8) || !lin_ok(cond->guid2, i8) || !lin_ok(cond->vec1, i8) ||
      !lin_ok(cond->vec2, i8))
    return MMDIT_ERR_ARG;
  const int D = d.D, C_txt = cond->C_txt, C_pool = cond->C_pool;
  if (C_txt <= 0 || C_txt % 64 || C_pool <= 0 || C_pool % 16) return MMDIT_ERR_SHAPE;
  if ((size_t)d.B * (C_pool > D ? C_pool : D) * 4 > 200 * 1024) return MMDIT_ERR_SHAPE;  // GEMV input in shared memory
  if (!al16(x_lat) || (txt && !al16(txt)) || !al16(pooled) || !al16(ws)) return MMDIT_ERR_ALIGN;
  size_t need = 0;
  MMDIT_TRY(mmdit_sample_workspace_size(shape, w->n_double, w->n_single, C_txt, n_steps, &need));
  if (ws_bytes < need) return MMDIT_ERR_WORKSPACE;
  MMDIT_TRY(check_device());
  cudaStream_t st = S(stream);
  Carve c{static_cast<uint8_t*>(ws), 0};
  StepWS sw;
  layout_step(d, *shape, w->n_double, w->n_single, c, sw);
  SampleWS sa;
  layout_sample(d, *shape, w->n_double, w->n_single, C_txt, n_steps, c, sa);

  // step-independent work: RoPE tables, the text stream, the conditioning vector
  MMDIT_CUDA(launch_rope_build(d.Lt, shape->grid_w, d.Lg, shape->ref_w, d.L, shape->rope_axes, shape->rope_theta,
                               nullptr, sw.cs, sw.sn, st));
  if (d.Lt > 0) {
    GemmParams p = gemm_params(GM_STORE_F32);
    p.out = sa.x_txt;
    p.out_ld = D;
    p.out_seg_rows = d.Lt;
    MMDIT_TRY(run_gemm(txt, C_txt, d.Lt, d.Lt, d.B, C_txt, cond->txt_in, D, p, sa.wdeq, st));
  }
  float* gh = sa.ctemb + (size_t)d.B * shape->t_dim;
  MMDIT_CUDA(launch_sinusoid(1000.0 * guidance, d.B, shape->t_dim, sa.ctemb, st));
  MMDIT_CUDA(launch_gemv(cond->guid1.w, i8, cond->guid1.scale, cond->guid1.b, sa.ctemb, d.B, D, shape->t_dim, 0, gh,
                         st));
  MMDIT_CUDA(launch_gemv(cond->guid2.w, i8, cond->guid2.scale, cond->guid2.b, gh, d.B, D, D, 1, sa.vec_cond, st));
  MMDIT_CUDA(launch_gemv(cond->vec1.w, i8, cond->vec1.scale, cond->vec1.b, pooled, d.B, D, C_pool, 0, sa.phid, st));
  MMDIT_CUDA(launch_gemv(cond->vec2.w, i8, cond->vec2.scale, cond->vec2.b, sa.phid, d.B, D, D, 1, sa.ptmp, st));
  MMDIT_CUDA(launch_add(sa.vec_cond, sa.ptmp, (long long)d.B * D, st));

  // Every step's conditioning vector vec_k = time2 SiLU(time1 sinusoid(1000 sigma_k)) + vec_cond, then the
  // modulation vectors of every step in one pass per sample: the modulation weights (the largest read of a
  // step after the block weights) are read once per 8 steps instead of once per step.
  {
    float* th = sw.temb + (size_t)d.B * shape->t_dim;
    for (int k = 0; k < n_steps; ++k) {
      MMDIT_CUDA(launch_sinusoid(1000.0 * sigmas[k], d.B, shape->t_dim, sw.temb, st));
      MMDIT_CUDA(launch_gemv(w->time1.w, w->time1.scale != nullptr, w->time1.scale, w->time1.b, sw.temb, d.B, D,
                             shape->t_dim, 0, th, st));
      MMDIT_CUDA(launch_gemv(w->time2.w, w->time2.scale != nullptr, w->time2.scale, w->time2.b, th, d.B, D, D, 1,
                             sw.vec, st));
      MMDIT_CUDA(launch_add(sw.vec, sa.vec_cond, (long long)d.B * D, st));
      MMDIT_CUDA(cudaMemcpy2DAsync(sa.vec_all + (size_t)k * D, (size_t)n_steps * D * 4, sw.vec, (size_t)D * 4,
                                   (size_t)D * 4, d.B, cudaMemcpyDeviceToDevice, st));
    }
    const long long mods_n = (long long)mods_floats(d, w->n_double, w->n_single);
    for (int b = 0; b < d.B; ++b) {
      // rows k of sample b: outputs at mods_all + k * mods_n, in the step buffer's layout at sample b
      std::vector<GemvJob> jobs = mod_jobs(d, *w, sa.mods_all, mods_n);
      size_t off = 0;
      for (GemvJob& j : jobs) {
        j.out = sa.mods_all + off + (size_t)b * j.N;
        off += (size_t)d.B * j.N;
      }
      MMDIT_CUDA(launch_gemv_batched(jobs.data(), (int)jobs.size(), i8, sa.vec_all + (size_t)b * n_steps * D,
                                     n_steps, D, 1, st));
    }
  }

  // step 0 eagerly (this also performs every one-time kernel set-up before a capture)
  MMDIT_TRY(step_impl(*shape, d, *w, x_lat, nullptr, sa.x_txt, sigmas[0], sigmas[1], nullptr, sa.vec_cond, nullptr,
                      nullptr, false, sw, st, sa.mods_all, 0));
  const bool graph = (flags & MMDIT_SAMPLE_GRAPH) && n_steps > 1 && !g_trace.on;
  if (!graph) {
    for (int i = 1; i < n_steps; ++i)
      MMDIT_TRY(step_impl(*shape, d, *w, x_lat, nullptr, sa.x_txt, sigmas[i], sigmas[i + 1], nullptr, sa.vec_cond,
                          nullptr, nullptr, false, sw, st, sa.mods_all, i));
    return MMDIT_OK;
  }
  // Steps 1 .. n - 1: one captured step reading sigma_k, sigma_{k+1} at the
  // device counter k, which the captured step advances at its end.
  MMDIT_CUDA(cudaMemcpyAsync(sa.sig, sigmas, sizeof(double) * ((size_t)n_steps + 1), cudaMemcpyHostToDevice, st));
  MMDIT_CUDA(launch_counter(sa.ctr, 1, false, st));
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return MMDIT_ERR_CUDA;
  cudaGraph_t graph_def = nullptr;
  cudaGraphExec_t exec = nullptr;
  int rc = MMDIT_OK;
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    rc = MMDIT_ERR_CUDA;
  } else {
    rc = step_impl(*shape, d, *w, x_lat, nullptr, sa.x_txt, 0.0, 0.0, nullptr, sa.vec_cond, sa.sig, sa.ctr, false, sw,
                   cs, sa.mods_all, 0);
    if (rc == MMDIT_OK) rc = cuda_status(launch_counter(sa.ctr, 1, true, cs));
    const cudaError_t e = cudaStreamEndCapture(cs, &graph_def);  // always closes the capture
    if (rc == MMDIT_OK && e != cudaSuccess) rc = MMDIT_ERR_CUDA;
  }
  if (rc == MMDIT_OK && cudaGraphInstantiate(&exec, graph_def, 0) != cudaSuccess) rc = MMDIT_ERR_CUDA;
  for (int i = 1; rc == MMDIT_OK && i < n_steps; ++i)
    if (cudaGraphLaunch(exec, st) != cudaSuccess) rc = MMDIT_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess && rc == MMDIT_OK) rc = MMDIT_ERR_CUDA;  // replays done
  if (exec) cudaGraphExecDestroy(exec);
  if (graph_def) cudaGraphDestroy(graph_def);
  cudaStreamDestroy(cs);
  return rc;
}

double mmdit_shift_mu(int n_image_tokens) {
  return 0.5 + ((double)n_image_tokens - 256.0) * (1.15 - 0.5) / (4096.0 - 256.0);
}

int mmdit_sigma_schedule(int n_steps, double mu, double* sigmas) {
  if (n_steps < 1 || !sigmas) return MMDIT_ERR_ARG;
  const double s = std::exp(mu);
  for (int i = 0; i <= n_steps; ++i) {
    const double t = 1.0 - (double)i / n_steps;
    sigmas[i] = s * t / (1.0 + (s - 1.0) * t);
  }
  return MMDIT_OK;
}

int mmdit_selftest_wait_timeout(unsigned limit_us, void* stream) {
  if (limit_us == 0 || limit_us > 1000000u) return MMDIT_ERR_ARG;
  MMDIT_TRY(check_device());
  return cuda_status(launch_wait_selftest(1000ull * limit_us, device_status_ptr(), S(stream)));
}

int euler_step(float* x, const void* v, int v_dtype, double sigma, double sigma_next, int64_t n, void* stream) {
  if (!x || !v || n < 0) return MMDIT_ERR_ARG;
  if (v_dtype != MMDIT_F32 && v_dtype != MMDIT_BF16) return MMDIT_ERR_ARG;
  if (!al16(x) || !al16(v)) return MMDIT_ERR_ALIGN;
  if (n == 0) return MMDIT_OK;
  MMDIT_TRY(check_device());
  return cuda_status(launch_euler(x, v, v_dtype == MMDIT_BF16, (float)(sigma_next - sigma), n, S(stream)));
}

int mmdit_heads_pack(const void* src, int64_t rows, int src_ld, int sections, int groups, int group_cols, void* dst,
                     void* stream) {
  if (!src || !dst || rows < 0 || sections < 1 || groups < 1) return MMDIT_ERR_ARG;
  if (group_cols < 8 || group_cols % 8 || src_ld % 8 || (long long)src_ld < (long long)sections * groups * group_cols)
    return MMDIT_ERR_SHAPE;
  if (!al16(src) || !al16(dst)) return MMDIT_ERR_ALIGN;
  if (rows == 0) return MMDIT_OK;
  MMDIT_TRY(check_device());
  return cuda_status(launch_heads_pack(static_cast<const uint16_t*>(src), rows, src_ld, sections, groups, group_cols,
                                       static_cast<uint16_t*>(dst), S(stream)));
}

int mmdit_heads_unpack(const void* src, int64_t rows, int groups, int group_cols, void* dst, int dst_ld,
                       void* stream) {
  if (!src || !dst || rows < 0 || groups < 1) return MMDIT_ERR_ARG;
  if (group_cols < 8 || group_cols % 8 || dst_ld % 8 || (long long)dst_ld < (long long)groups * group_cols)
    return MMDIT_ERR_SHAPE;
  if (!al16(src) || !al16(dst)) return MMDIT_ERR_ALIGN;
  if (rows == 0) return MMDIT_OK;
  MMDIT_TRY(check_device());
  return cuda_status(launch_heads_unpack(static_cast<const uint16_t*>(src), rows, groups, group_cols,
                                         static_cast<uint16_t*>(dst), dst_ld, S(stream)));
}

int mmdit_quantize_w8(const void* w, int w_dtype, int N, int K, int8_t* q, float* scale, void* stream) {
  if (!w || !q || !scale) return MMDIT_ERR_ARG;
  if (w_dtype != MMDIT_F32 && w_dtype != MMDIT_BF16) return MMDIT_ERR_ARG;
  if (N < 1 || K < 1) return MMDIT_ERR_SHAPE;
  MMDIT_TRY(check_device());
  return cuda_status(launch_quantize(w, w_dtype == MMDIT_BF16, N, K, q, scale, S(stream)));
}

int mmdit_quantize_f8(const void* x, int x_dtype, long long rows, int K, long long ld, uint8_t* q, float* s,
                      void* stream) {
  if (!x || !q || !s || rows < 0 || K < 2 || K % 2 || ld < K) return MMDIT_ERR_ARG;
  if (x_dtype != MMDIT_BF16 && x_dtype != MMDIT_F32) return MMDIT_ERR_ARG;
  if (rows > (1ll << 31) - 1) return MMDIT_ERR_SHAPE;
  if (rows == 0) return MMDIT_OK;
  MMDIT_TRY(check_device());
  return cuda_status(launch_quantize_f8(x, x_dtype == MMDIT_BF16, rows, K, ld, q, K, s, S(stream)));
}

// The GEMM epilogue parameters of the test hooks' epilogue codes (y has N
// columns; N / 2 for SwiGLU).
static int linear_epilogue(int epilogue, int M, int N, void* y, const float* gate, GemmParams& p) {
  switch (epilogue) {
    case MMDIT_EPI_BF16:
    case MMDIT_EPI_BF16_GELU:
      p = gemm_params(GM_STORE_BF16);
      if (epilogue == MMDIT_EPI_BF16_GELU) p.gelu_from = 0;
      p.out = y;
      p.out_ld = N;
      p.out_seg_rows = M;
      return MMDIT_OK;
    case MMDIT_EPI_F32:
      p = gemm_params(GM_STORE_F32);
      p.out = y;
      p.out_ld = N;
      p.out_seg_rows = M;
      return MMDIT_OK;
    case MMDIT_EPI_SWIGLU:
      p = gemm_params(GM_SWIGLU);
      p.out = y;
      p.out_ld = N / 2;
      p.out_seg_rows = M;
      return MMDIT_OK;
    case MMDIT_EPI_RESID:
      p = gemm_params(GM_RESID);
      p.resid = static_cast<float*>(y);
      p.resid_ld = N;
      p.resid_seg_rows = M;
      p.gate = gate;
      p.gate_seg_stride = 0;
      return MMDIT_OK;
    default:
      return MMDIT_ERR_ARG;
  }
}

int mmdit_linear_f8_fwd(const mmdit_linear_t* lin, int M, int N, int K, const uint8_t* x, const float* x_scale,
                        void* y, int epilogue, const float* gate, void* stream) {
  if (!lin || !lin->w || !lin->scale || !x || !x_scale || !y) return MMDIT_ERR_ARG;
  if (M < 1 || N < 32 || N % 32 || K < 128 || K % 128) return MMDIT_ERR_SHAPE;
  if (!al16(x) || !al16(y) || !al16(lin->w) || !al16(lin->scale) || (lin->b && !al16(lin->b)) ||
      (gate && !al16(gate)))
    return MMDIT_ERR_ALIGN;
  GemmParams p;
  MMDIT_TRY(linear_epilogue(epilogue, M, N, y, gate, p));
  MMDIT_TRY(check_device());
  p.ascale = x_scale;
  return run_gemm(x, K, M, M, 1, K, *lin, N, p, nullptr, S(stream));
}

int mmdit_linear_fwd(const mmdit_linear_t* lin, int M, int N, int K, const void* x, void* y, int epilogue,
                     const float* gate, void* ws, size_t ws_bytes, void* stream) {
  if (!lin || !x || !y) return MMDIT_ERR_ARG;
  if (!lin_ok(*lin, lin->scale != nullptr)) return MMDIT_ERR_ARG;
  if (M < 1 || N < 32 || N % 32 || K < 64 || K % 64) return MMDIT_ERR_SHAPE;
  if (!al16(x) || !al16(y) || (gate && !al16(gate))) return MMDIT_ERR_ALIGN;
  uint16_t* wdeq = nullptr;
  if (lin->scale) {
    if (!ws || ws_bytes < (size_t)N * K * 2) return MMDIT_ERR_WORKSPACE;
    if (!al16(ws)) return MMDIT_ERR_ALIGN;
    wdeq = static_cast<uint16_t*>(ws);
  }
  GemmParams p;
  MMDIT_TRY(linear_epilogue(epilogue, M, N, y, gate, p));
  MMDIT_TRY(check_device());
  return run_gemm(x, K, M, M, 1, K, *lin, N, p, wdeq, S(stream));
}

int mmdit_ln_modulate(const float* x, int B, int rows, int D, const float* shift, const float* scale,
                      int64_t mod_stride, float eps, void* y, void* stream) {
  if (!x || !shift || !scale || !y) return MMDIT_ERR_ARG;
  if (B < 1 || rows < 1 || D < 256 || D % 256 || D > 4096) return MMDIT_ERR_SHAPE;
  if (!al16(x) || !al16(shift) || !al16(scale) || !al16(y) || (mod_stride % 4)) return MMDIT_ERR_ALIGN;
  MMDIT_TRY(check_device());
  return cuda_status(
      launch_ln_modulate(x, rows, rows, B, D, shift, scale, mod_stride, eps, static_cast<uint16_t*>(y), S(stream)));
}

int mmdit_ln_modulate_f8(const float* x, int B, int rows, int D, const float* shift, const float* scale,
                         int64_t mod_stride, float eps, void* y, uint8_t* q, float* s, void* stream) {
  if (!x || !shift || !scale || !q || !s) return MMDIT_ERR_ARG;
  if (B < 1 || rows < 1 || D < 256 || D % 256 || D > 4096) return MMDIT_ERR_SHAPE;
  if (!al16(x) || !al16(shift) || !al16(scale) || (y && !al16(y)) || !al16(q) || !al16(s) || (mod_stride % 4))
    return MMDIT_ERR_ALIGN;
  MMDIT_TRY(check_device());
  return cuda_status(launch_ln_modulate(x, rows, rows, B, D, shift, scale, mod_stride, eps, static_cast<uint16_t*>(y),
                                        S(stream), q, s));
}

int mmdit_gemv(const mmdit_linear_t* lin, int B, int N, int K, const float* x, int act, float* y, void* stream) {
  if (!lin || !x || !y || (act != 0 && act != 1)) return MMDIT_ERR_ARG;
  if (!lin_ok(*lin, lin->scale != nullptr)) return MMDIT_ERR_ARG;
  if (B < 1 || B > 16 || N < 1 || K < 16 || K % 16) return MMDIT_ERR_SHAPE;
  if ((size_t)8 * K * 4 > 200 * 1024) return MMDIT_ERR_SHAPE;  // 8 rows of x in shared memory
  MMDIT_TRY(check_device());
  return cuda_status(launch_gemv(lin->w, lin->scale != nullptr, lin->scale, lin->b, x, B, N, K, act, y, S(stream)));
}

int mmdit_time_embed(const mmdit_shape_t* shape, const mmdit_linear_t* time1, const mmdit_linear_t* time2,
                     double sigma, float* vec, float* ws, void* stream) {
  Dims d;
  MMDIT_TRY(check_shape(shape, &d));
  if (!time1 || !time2 || !vec || !ws) return MMDIT_ERR_ARG;
  if (shape->t_dim <= 0 || shape->t_dim % 16) return MMDIT_ERR_SHAPE;
  if (!lin_ok(*time1, time1->scale != nullptr) || !lin_ok(*time2, time2->scale != nullptr)) return MMDIT_ERR_ARG;
  if (!al16(vec) || !al16(ws)) return MMDIT_ERR_ALIGN;
  MMDIT_TRY(check_device());
  cudaStream_t st = S(stream);
  MMDIT_CUDA(launch_sinusoid(1000.0 * sigma, d.B, shape->t_dim, ws, st));
  float* th = ws + (size_t)d.B * shape->t_dim;
  MMDIT_CUDA(launch_gemv(time1->w, time1->scale != nullptr, time1->scale, time1->b, ws, d.B, d.D, shape->t_dim, 0,
                         th, st));
  return cuda_status(
      launch_gemv(time2->w, time2->scale != nullptr, time2->scale, time2->b, th, d.B, d.D, d.D, 1, vec, st));
}

}  // extern "C"
