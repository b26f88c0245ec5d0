/*
 * mmdit.h - C ABI of a GB300 (sm_103a) library for the forward pass of one
 * Flux-style multi-modal diffusion transformer (MMDiT) denoising step.
 *
 * Sources.  The operations follow the primitive definitions in the Luminal
 * blog post "Reducing image generation cost with ..." (section "What the
 * compiler found on its own": matmul, attention as scores/scale/max/exp/
 * sum/divide, RMSNorm, LayerNorm, adaLN scale-and-shift, RoPE as a partner
 * gather with cosine/sine tables, gate-and-residual add, text/image
 * concatenation, timestep embedding), the block structure of its section
 * "Flux.2 Klein 9B" (double-stream and single-stream blocks, 16x latent
 * patches with 128 channels), the host-side Euler sampler of its section
 * "The AMD MI300X pipeline", and the int8 weight-only setting of the
 * flux-amd-rocm BENCHMARKS.md page (torchao Int8WeightOnlyConfig).  Readings
 * of steps the pages leave open are stated at each declaration.
 *
 * Conventions shared by every entry point:
 *  - Return value: MMDIT_OK (0) or a negative MMDIT_ERR_* code.  On an
 *    argument error nothing is launched.  Launches are asynchronous on the
 *    given stream (a cudaStream_t passed as void*; NULL = legacy default).
 *    A kernel that gives up a bounded wait records MMDIT_ERR_TIMEOUT in a
 *    device status word that mmdit_sync_status() reads and clears.
 *  - Pointers marked "device" must be device memory, owned by the caller,
 *    and 16-byte aligned.  The library allocates no device memory: scratch
 *    comes from the caller's workspace, sized by mmdit_workspace_size().
 *  - Tensors are dense row-major.  bf16 = IEEE bfloat16 bits (uint16).
 *    Linear weights are [N_out, K_in] row-major (y = x W^T + b), bias fp32
 *    [N_out].  Int8 weights are int8 [N_out, K_in] with an fp32 per-row
 *    scale: W = q * scale[n].
 *  - Token layout: per sample, the L_txt text tokens come first, then the
 *    L_img = grid_h * grid_w image tokens in row-major (h, w) order; the
 *    batch index is outermost.
 *  - The residual streams are fp32 and are updated in place.  GEMM and
 *    attention operands are bf16 with fp32 accumulation; norms, softmax and
 *    modulation are computed in fp32.
 *  - Limits: D a multiple of 256, d_head 64 or 128, H * d_head == D,
 *    D_mlp a multiple of 64, rope_axes summing to d_head with even entries,
 *    1 <= B, L_txt >= 0, L_img >= 1.
 */
#ifndef MMDIT_H_
#define MMDIT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status */
#define MMDIT_OK 0
#define MMDIT_ERR_ARG (-1)         /* null pointer or bad enum value */
#define MMDIT_ERR_SHAPE (-2)       /* shape outside the limits above */
#define MMDIT_ERR_ALIGN (-3)       /* pointer or stride not 16-byte aligned */
#define MMDIT_ERR_WORKSPACE (-4)   /* workspace smaller than required */
#define MMDIT_ERR_CUDA (-5)        /* a CUDA runtime call failed */
#define MMDIT_ERR_TIMEOUT (-6)     /* a kernel abandoned a bounded wait */
#define MMDIT_ERR_UNSUPPORTED (-7) /* device is not sm_103 / feature absent */

/* ---------------------------------------------------------------- dtypes */
#define MMDIT_BF16 0
#define MMDIT_F32 1
#define MMDIT_I8W 2 /* int8 weight with fp32 per-output-channel scale */
/* e4m3 weights with fp32 per-output-channel scales for the block GEMMs (qkv,
 * proj, mlp_in, mlp_out, lin1, lin2: mmdit_quantize_f8 codes), their
 * activations quantised to e4m3 per row on the fly, tcgen05 kind::f8f6f4
 * MMAs; modulation and step-level linears stay bf16 (scale NULL). */
#define MMDIT_F8W 3

/* ---------------------------------------------------------------- shapes */
typedef struct {
  int B;            /* batch (independent samples) */
  int L_txt;        /* text tokens per sample */
  int grid_h;       /* latent grid rows */
  int grid_w;       /* latent grid columns; L_img = grid_h * grid_w */
  int D;            /* hidden width */
  int H;            /* attention heads */
  int d_head;       /* head width (64 or 128) */
  int D_mlp;        /* MLP hidden width */
  int rope_axes[3]; /* channels per RoPE axis (id, row, column) */
  double rope_theta;
  float eps_ln;     /* LayerNorm epsilon */
  float eps_rms;    /* q/k RMSNorm epsilon */
  int w_dtype;      /* MMDIT_BF16, MMDIT_I8W (all linears) or MMDIT_F8W (block GEMM linears) */
  int C_lat;        /* latent channels per image token (step only) */
  int t_dim;        /* timestep sinusoid width (step only) */
  int mlp_act;      /* MMDIT_MLP_GELU or MMDIT_MLP_SWIGLU (see below) */
  int ref_h;        /* reference latent grid rows (image-to-image), 0 = none */
  int ref_w;        /* reference latent grid columns, 0 = none */
} mmdit_shape_t;

/* Reference latent (image-to-image).  The Luminal blog (section "The AMD
 * MI300X pipeline") computes the reference image's latent once per run and
 * appends it to the noise tokens; no page gives its positions.  Reading
 * taken: per sample the tokens are [text (L_txt); target image (grid_h x
 * grid_w, row-major); reference image (ref_h x ref_w, row-major)], and the
 * RoPE position of a token is text (0, 0, 0), target (0, h, w), reference
 * (1, h, w): the reference sits on its own grid and differs from the target
 * on the first axis, which text and target leave at 0.  The blocks treat all
 * image tokens alike: the image stream of a double block holds
 * L_img = grid_h grid_w + ref_h ref_w tokens per sample, in this order.  The
 * step (mmdit_step_i2i_fwd) projects both latents with img_in and applies
 * the final layer and the Euler update to the target tokens only.  ref_h and
 * ref_w are both 0 or both positive. */

/* MLP activation.  GELU-tanh: mlp_in (double) and the MLP rows of lin1
 * (single) have D_mlp output rows.  SwiGLU (the Flux.2 Klein blocks; the
 * Luminal blog, section "What the compiler found on its own", lists the
 * SwiGLU activation among the fused kernels of a Klein step): they have
 * 2 D_mlp rows [gate; up] and the activation is SiLU(gate) * up, D_mlp
 * wide (D_mlp a multiple of 128). */
#define MMDIT_MLP_GELU 0
#define MMDIT_MLP_SWIGLU 1

/* One linear layer.  w: device [N, K] (bf16, or int8 when scale != NULL);
 * b: device fp32 [N] or NULL; scale: device fp32 [N] for int8 weights. */
typedef struct {
  const void* w;
  const float* b;
  const float* scale;
} mmdit_linear_t;

/* Double-stream block weights; index 0 = text stream, 1 = image stream.
 * mod: D -> 6D, chunks (shift1, scale1, gate1, shift2, scale2, gate2).
 * qkv: D -> 3D (q | k | v, head-major inside each).  proj: D -> D.
 * mlp_in: D -> D_mlp (GELU-tanh).  mlp_out: D_mlp -> D.
 * q_norm / k_norm: device fp32 [d_head] RMSNorm gains. */
typedef struct {
  mmdit_linear_t mod[2], qkv[2], proj[2], mlp_in[2], mlp_out[2];
  const float* q_norm[2];
  const float* k_norm[2];
} mmdit_double_w_t;

/* Single-stream block weights.  mod: D -> 3D (shift, scale, gate).
 * lin1: D -> 3D + D_mlp (q | k | v | mlp).  lin2: D + D_mlp -> D over
 * [attention output | GELU-tanh(mlp)]. */
typedef struct {
  mmdit_linear_t mod, lin1, lin2;
  const float* q_norm;
  const float* k_norm;
} mmdit_single_w_t;

/* Whole-step weights.  time1: t_dim -> D, time2: D -> D (SiLU between);
 * img_in: C_lat -> D; final_mod: D -> 2D (shift, scale); final: D -> C_lat. */
typedef struct {
  mmdit_linear_t time1, time2, img_in, final_mod, final;
  const mmdit_double_w_t* doubles; /* host array of n_double */
  int n_double;
  const mmdit_single_w_t* singles; /* host array of n_single */
  int n_single;
} mmdit_step_w_t;

/* ------------------------------------------------------------ utilities */
const char* mmdit_status_string(int status);

/* Synchronises `stream`, then reads and clears the device status word of
 * the current device.  Returns MMDIT_ERR_TIMEOUT if a kernel abandoned a
 * bounded wait since the last call, MMDIT_ERR_CUDA on a sticky CUDA error. */
int mmdit_sync_status(void* stream);

/* Failure-detection self-test: launches one tiny kernel that waits on a
 * barrier nothing ever completes, with a limit of limit_us microseconds
 * (1 .. 1e6).  The wait gives up, records its bit in the device status word
 * and the kernel returns normally; the next mmdit_sync_status() reports
 * MMDIT_ERR_TIMEOUT and clears the word.  No fault, trap or hang. */
int mmdit_selftest_wait_timeout(unsigned limit_us, void* stream);

/* Number of kernels this library has launched in this process. */
long long mmdit_launch_count(void);

/* Launch trace.  mmdit_trace_begin creates 2*capacity CUDA events (call it
 * outside stream capture) and turns tracing on: each of the next `capacity`
 * kernel launches is bracketed by an event pair on its own stream.
 * mmdit_trace_end turns it off and reports how many launches were recorded;
 * mmdit_trace_read waits for them and returns each launch's kernel id and
 * duration in milliseconds.  mmdit_kernel_name maps an id to a name. */
int mmdit_trace_begin(int capacity);
int mmdit_trace_end(int* count);
int mmdit_trace_read(int* kernel_ids, float* ms, int capacity, int* count);
const char* mmdit_kernel_name(int kernel_id);

/* Workspace bytes the named operation needs for `shape` (vec given, i.e.
 * the block computes its own modulation).
 * op: MMDIT_OP_DOUBLE, MMDIT_OP_SINGLE or MMDIT_OP_ATTENTION. */
#define MMDIT_OP_DOUBLE 1
#define MMDIT_OP_SINGLE 2
#define MMDIT_OP_ATTENTION 3
int mmdit_workspace_size(const mmdit_shape_t* shape, int op, size_t* bytes);

/* Workspace bytes of mmdit_step_fwd for n_double + n_single blocks
 * (C_lat a multiple of 64, t_dim a multiple of 16). */
int mmdit_step_workspace_size(const mmdit_shape_t* shape, int n_double, int n_single, size_t* bytes);

/* ------------------------------------------------------------ RoPE */
/* Position ids and rotation tables for 2D axial RoPE.
 * The Luminal blog (section "What the compiler found on its own") describes
 * RoPE as pairing each channel with a partner channel and combining the two
 * with cosine and sine tables; it fixes nothing else.  Reading taken: text
 * token i sits at (0, 0, 0); target image token (h, w) at (0, h, w); a
 * reference image token (h, w) at (1, h, w).  Channel pairs are adjacent, (2i, 2i+1); the
 * first rope_axes[0]/2 pairs follow axis 0, the next rope_axes[1]/2 axis 1,
 * the rest axis 2.  Pair i of axis a turns by pos_a * theta^(-2i/rope_axes[a]),
 * computed in fp64 and rounded once to fp32.
 * ids: device int32 [L, 3]; cos_, sin_: device fp32 [L, d_head/2]. */
int mmdit_rope2d_build(const mmdit_shape_t* shape, int32_t* ids, float* cos_, float* sin_, void* stream);

/* Rotates x in place: x device bf16 [B, L, H, d_head] with token row stride
 * `row_stride` elements (>= H*d_head, multiple of 8):
 * (x0, x1) -> (x0 c - x1 s, x0 s + x1 c) per pair, in fp32. */
int rope2d_apply(const mmdit_shape_t* shape, const float* cos_, const float* sin_, void* x, int row_stride,
                 void* stream);

/* ------------------------------------------------------------ attention */
/* Joint softmax attention over the concatenated [text; image] sequence of
 * each sample, one softmax per (sample, head, query), scale 1/sqrt(d_head),
 * no mask (Luminal blog: attention = scores, scale, max, exp, sum, divide).
 * qkv: device bf16 [B, L, 3, H, d_head] with token row stride
 * `qkv_row_stride` elements (>= 3*D, multiple of 8).
 * q_norm / k_norm: device fp32 [d_head] gains; entry [0] applies to text
 * tokens, [1] to image tokens (pass the same pointer twice for one stream).
 * If q_norm[0] is NULL no RMSNorm is applied; if cos_ is NULL no RoPE.
 * Otherwise q and k get RMSNorm (eps_rms) and then RoPE before the scores.
 * out: device bf16 [B, L, H*d_head], token row stride out_row_stride.
 * ws: device workspace of mmdit_workspace_size(MMDIT_OP_ATTENTION) bytes. */
int joint_attention_fwd(const mmdit_shape_t* shape, const void* qkv, int qkv_row_stride, const float* const q_norm[2],
                        const float* const k_norm[2], const float* cos_, const float* sin_, void* out,
                        int out_row_stride, void* ws, size_t ws_bytes, void* stream);

/* joint_attention_fwd for callers that cannot allocate device memory.
 * No counterpart on the pages: this is a deployment variant.  A caller such
 * as a plugin inside a host application that owns every device allocation,
 * or code that must avoid the implicit synchronisation cudaMalloc/cudaFree
 * can cause, may have no workspace to pass.  This call computes the
 * attention joint_attention_fwd computes (same arguments minus ws/ws_bytes)
 * and allocates nothing: its scratch is a fixed 48 MiB device array inside
 * the library, reserved on every GPU that loads it until the process exits.
 *  - The scratch holds the normalised, rotated q and k (B*L*2*D bf16) and
 *    the transposed v (B*D*Lpad bf16, Lpad = L rounded up to 8), each
 *    256-byte aligned.  Shapes needing more than 48 MiB return
 *    MMDIT_ERR_WORKSPACE and launch nothing.
 *  - With at most one work unit (a pair of 128-row query tiles of one
 *    sample and head) per SM the result is bit-identical to
 *    joint_attention_fwd's.  Above that, joint_attention_fwd balances its
 *    last rounds by splitting units in two and merging the parts, which
 *    this call (no merge area) does not, so the two may differ by rounding.
 *  - The array is shared by all calls on a device: calls that overlap on
 *    the GPU (e.g. on two streams) race.  It keeps the last call's contents;
 *    nothing in it needs clearing, since each call writes every byte it reads.
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture. */
int joint_attention_fwd_noalloc(const mmdit_shape_t* shape, const void* qkv, int qkv_row_stride,
                                const float* const q_norm[2], const float* const k_norm[2], const float* cos_,
                                const float* sin_, void* out, int out_row_stride, void* stream);

/* ------------------------------------------------------------ blocks */
/* Double-stream block, in place on x_txt (device fp32 [B, L_txt, D]) and
 * x_img (device fp32 [B, L_img, D]).  vec: device fp32 [B, D] conditioning
 * vector; or pass vec = NULL and mod_precomputed = device fp32 [2, B, 6D]
 * (stream, sample, chunk) already equal to mod.W SiLU(vec) + mod.b.
 * Per stream: y = LN(x)(1 + scale1) + shift1; q, k, v = y Wqkv^T + b;
 * q, k <- RMSNorm then RoPE; o = joint attention; x += gate1 (o Wp^T + bp);
 * y2 = LN(x)(1 + scale2) + shift2; x += gate2 (GELU(y2 W1^T + b1) W2^T + b2).
 * cos_/sin_: tables from mmdit_rope2d_build. */
int mmdit_double_block_fwd(const mmdit_shape_t* shape, const mmdit_double_w_t* w, const float* vec,
                           const float* mod_precomputed, float* x_txt, float* x_img, const float* cos_,
                           const float* sin_, void* ws, size_t ws_bytes, void* stream);

/* Single-stream block, in place on x (device fp32 [B, L, D], text first).
 * mod_precomputed, if used: device fp32 [B, 3D].
 * y = LN(x)(1 + scale) + shift; [q k v m] = y W1^T + b1; q, k <- RMSNorm,
 * RoPE; x += gate ([attention(q,k,v) | GELU(m)] W2^T + b2). */
int mmdit_single_block_fwd(const mmdit_shape_t* shape, const mmdit_single_w_t* w, const float* vec,
                           const float* mod_precomputed, float* x, const float* cos_, const float* sin_, void* ws,
                           size_t ws_bytes, void* stream);

/* ------------------------------------------------------------ step */
/* One denoising step: vec = time2 SiLU(time1 sinusoid(1000 sigma) + b) + b;
 * x_img = img_in(x_lat); the n_double double blocks on (x_txt_in, x_img);
 * the n_single single blocks on [x_txt; x_img]; v = final(LN(x_img)(1 +
 * scale) + shift); x_lat += (sigma_next - sigma) v.
 * The sinusoid has t_dim/2 frequencies 10000^(-j/(t_dim/2)), order [cos | sin].
 * x_lat: device fp32 [B, L_img, C_lat], updated in place.
 * x_txt_in: device fp32 [B, L_txt, D], read only.
 * v_out: device fp32 [B, L_img, C_lat] or NULL. */
int mmdit_step_fwd(const mmdit_shape_t* shape, const mmdit_step_w_t* w, float* x_lat, const float* x_txt_in,
                   double sigma, double sigma_next, float* v_out, void* ws, size_t ws_bytes, void* stream);

/* The same step with a reference latent (shape->ref_h, ref_w > 0): the image
 * tokens are img_in([x_lat; x_ref]) per sample, laid out as above.
 * x_lat: device fp32 [B, grid_h grid_w, C_lat], updated in place (target
 * tokens only).  x_ref: device fp32 [B, ref_h ref_w, C_lat], read only.
 * v_out: device fp32 [B, grid_h grid_w, C_lat] or NULL.  mmdit_step_fwd is
 * this call without a reference (it rejects ref_h > 0 with MMDIT_ERR_ARG;
 * so does mmdit_sample). */
int mmdit_step_i2i_fwd(const mmdit_shape_t* shape, const mmdit_step_w_t* w, float* x_lat, const float* x_ref,
                       const float* x_txt_in, double sigma, double sigma_next, float* v_out, void* ws,
                       size_t ws_bytes, void* stream);

/* ------------------------------------------------------------ sequence parallelism */
/* Exchange layouts of Ulysses sequence parallelism.  The SGLang blog
 * ("Architecture Deep Dive", "SGLang Diffusion Serving") scales the DiT over
 * several GPUs with USP, hybrid Ulysses sequence parallelism and ring
 * attention; Ulysses gives each of P ranks a shard of the token sequence for
 * the linears and, around attention, swaps it for all tokens of H / P heads
 * with two all-to-all exchanges.  These calls lay the data out for those
 * exchanges on one device; the exchanges themselves belong to the caller's
 * collective library.  All data bf16, pointers device and 16-byte aligned,
 * group_cols and the row strides multiples of 8; no workspace.
 * mmdit_heads_pack: src [rows][src_ld] whose first sections * groups *
 * group_cols columns hold `sections` blocks (q | k | v) of `groups` head
 * groups of group_cols columns each; writes dst [groups][rows][sections]
 * [group_cols], the chunk for head group g contiguous at g * rows * sections
 * * group_cols.
 * mmdit_heads_unpack: src [groups][rows][group_cols] -> dst [rows][dst_ld],
 * head group g at columns g * group_cols .. (g + 1) * group_cols.
 * Errors: MMDIT_ERR_ARG (null pointer, counts below 1), MMDIT_ERR_SHAPE
 * (widths), MMDIT_ERR_ALIGN; nothing is launched then. */
int mmdit_heads_pack(const void* src, int64_t rows, int src_ld, int sections, int groups, int group_cols, void* dst,
                     void* stream);
int mmdit_heads_unpack(const void* src, int64_t rows, int groups, int group_cols, void* dst, int dst_ld,
                       void* stream);

/* ------------------------------------------------------------ sigma schedule */
/* The sampler's noise levels.  The Luminal blog (section "The AMD MI300X
 * pipeline") integrates the latent with an Euler sampler, and the flux-amd-rocm
 * benchmark notes run 28 steps; no page prints the schedule.  Reading taken
 * (the shifted-linear schedule of Flux-style models): t_i = 1 - i / n_steps,
 * sigma_i = s t_i / (1 + (s - 1) t_i) with s = exp(mu), i = 0 .. n_steps, so
 * sigma_0 = 1, sigma_n = 0; mu is linear in the image-token count through
 * (256, 0.5) and (4096, 1.15).  Host arithmetic in double precision; no
 * device work, callable without a GPU.
 * mmdit_shift_mu: mu for n_image_tokens (any value; no error case).
 * mmdit_sigma_schedule: writes sigmas[0 .. n_steps] (host array of n_steps + 1
 * doubles, caller-owned); MMDIT_ERR_ARG for n_steps < 1 or a NULL array. */
double mmdit_shift_mu(int n_image_tokens);
int mmdit_sigma_schedule(int n_steps, double mu, double* sigmas);

/* ------------------------------------------------------------ sampling loop */
/* Conditioning around the denoiser.  The SGLang blog ("Architecture") has a
 * text encoder produce the conditioning embeddings that the DiT denoises
 * against over 20-50 steps; the flux-amd-rocm benchmark notes sample
 * FLUX.1-dev for 28 steps at guidance 3.5.  Neither defines the layers;
 * readings taken: txt_in is one linear projection C_txt -> D of the
 * text-encoder output; the guidance scale g goes through the timestep's
 * sinusoid of 1000 g and a two-layer SiLU MLP (guid1: t_dim -> D,
 * guid2: D -> D); the pooled text vector y through vec1: C_pool -> D, SiLU,
 * vec2: D -> D.  Both MLP outputs are added to the timestep embedding of
 * every step.  Weights follow shape->w_dtype like the step's.
 * C_txt a multiple of 64, C_pool a multiple of 16. */
typedef struct {
  mmdit_linear_t txt_in, guid1, guid2, vec1, vec2;
  int C_txt, C_pool;
} mmdit_cond_w_t;

/* Replay the step through one captured CUDA graph (see mmdit_sample). */
#define MMDIT_SAMPLE_GRAPH 1

/* Workspace bytes of mmdit_sample for the given block counts, text width
 * and number of steps. */
int mmdit_sample_workspace_size(const mmdit_shape_t* shape, int n_double, int n_single, int C_txt, int n_steps,
                                size_t* bytes);

/* The sampling loop over sigmas[0 .. n_steps] (host array, fp64).
 * x_txt = txt_in(txt) and vec_cond = guid2 SiLU(guid1 sinusoid(1000
 * guidance)) + vec2 SiLU(vec1 pooled) are formed once; then for i = 0 ..
 * n_steps - 1 the step of mmdit_step_fwd runs with sigma_i, sigma_{i+1}
 * and vec_cond added to its timestep embedding, updating x_lat in place.
 * x_lat: device fp32 [B, L_img, C_lat]; txt: device bf16 [B, L_txt, C_txt]
 * (ignored when L_txt = 0); pooled: device fp32 [B, C_pool].
 * flags & MMDIT_SAMPLE_GRAPH: step 0 runs eagerly, steps 1 .. n_steps - 1
 * replay one captured graph of a step that reads its sigmas from the
 * workspace on the device (bit-identical results); the call then returns
 * only after the replays complete, and falls back to eager launches while
 * a kernel trace is being recorded.  Without the flag the call only
 * enqueues work on `stream`. */
int mmdit_sample(const mmdit_shape_t* shape, const mmdit_step_w_t* w, const mmdit_cond_w_t* cond, float* x_lat,
                 const void* txt, const float* pooled, double guidance, const double* sigmas, int n_steps, int flags,
                 void* ws, size_t ws_bytes, void* stream);

/* Flow-matching Euler update (Luminal blog, "The AMD MI300X pipeline": the
 * sampler integrates the latent in fp32): x[i] += (sigma_next - sigma) v[i].
 * x: device fp32 [n]; v: device [n], v_dtype MMDIT_F32 or MMDIT_BF16.
 * The step size is rounded once to fp32. */
int euler_step(float* x, const void* v, int v_dtype, double sigma, double sigma_next, int64_t n, void* stream);

/* ------------------------------------------------------------ int8 */
/* Per-output-channel symmetric int8 quantiser (flux-amd-rocm BENCHMARKS.md:
 * torchao Int8WeightOnlyConfig).  Reading: s_n = max_k |w_nk| / 127 in fp32
 * (1 for an all-zero row); q = clamp(rint(w / s_n), -127, 127), division
 * in fp32, ties to even.  w: device [N, K] of w_dtype (MMDIT_BF16 or
 * MMDIT_F32); q: device int8 [N, K]; scale: device fp32 [N]. */
int mmdit_quantize_w8(const void* w, int w_dtype, int N, int K, int8_t* q, float* scale, void* stream);

/* ------------------------------------------------------------ pieces */
/* Building blocks of the step, exported for tests and for callers that
 * compose their own loop. */

/* y = x W^T (+ b), x device bf16 [M, K]; epilogue:
 *   MMDIT_EPI_BF16:        y device bf16 [M, N]
 *   MMDIT_EPI_BF16_GELU:   y device bf16 [M, N], GELU-tanh applied
 *   MMDIT_EPI_F32:         y device fp32 [M, N]
 *   MMDIT_EPI_SWIGLU:      W rows [gate; up] (N a multiple of 256): y device bf16
 *                          [M, N/2] = SiLU(x Wg^T + bg) * (x Wu^T + bu)
 *   MMDIT_EPI_RESID:       y device fp32 [M, N] += gate[n] * (x W^T + b),
 *                          gate device fp32 [N] (NULL = 1)
 * Int8 weights when lin->scale != NULL (y = (x q^T) * scale + b); they are
 * widened to bf16 (exactly) in `ws`, which then needs N*K*2 bytes.
 * K a multiple of 64, N a multiple of 32. */
/* FP8 (e4m3) row quantiser.  The SGLang blog ("Architecture") names FP8
 * quantisation for serving without fixing a scheme; reading taken: each row
 * (an output channel of a weight, or an activation row) gets s = max|row| /
 * 448 (fp32; 1 for a zero row) and q = e4m3(x / s), the quotient rounded
 * once in fp32, then to the nearest e4m3 (ties to even, saturating at 448).
 * x: device [rows, K] with row stride ld elements, x_dtype MMDIT_BF16 or
 * MMDIT_F32; q: device e4m3 bytes [rows, K] (row stride K); s: device fp32
 * [rows].  K even. */
int mmdit_quantize_f8(const void* x, int x_dtype, long long rows, int K, long long ld, uint8_t* q, float* s,
                      void* stream);

/* y = (x (.) sx) (W (.) sw)^T + b on e4m3 operands (tcgen05 kind::f8f6f4,
 * fp32 accumulation): x device e4m3 [M, K] with row scales x_scale [M], W
 * (lin->w) e4m3 [N, K] with channel scales lin->scale [N] (required).
 * Epilogues and y as for mmdit_linear_fwd.  K a multiple of 128. */
int mmdit_linear_f8_fwd(const mmdit_linear_t* lin, int M, int N, int K, const uint8_t* x, const float* x_scale,
                        void* y, int epilogue, const float* gate, void* stream);

#define MMDIT_EPI_BF16 0
#define MMDIT_EPI_BF16_GELU 1
#define MMDIT_EPI_F32 2
#define MMDIT_EPI_RESID 3
#define MMDIT_EPI_SWIGLU 4
int mmdit_linear_fwd(const mmdit_linear_t* lin, int M, int N, int K, const void* x, void* y, int epilogue,
                     const float* gate, void* ws, size_t ws_bytes, void* stream);

/* y = LN(x)(1 + scale) + shift per row, x device fp32 [B, rows, D],
 * shift/scale device fp32 with sample stride mod_stride elements,
 * y device bf16 [B, rows, D]. */
int mmdit_ln_modulate(const float* x, int B, int rows, int D, const float* shift, const float* scale,
                      int64_t mod_stride, float eps, void* y, void* stream);

/* mmdit_ln_modulate followed by the e4m3 row quantisation of its bf16 result
 * (the activation path of MMDIT_F8W), in one pass: q device e4m3 bytes
 * [B, rows, D], s device fp32 [B, rows] with s = max|bf16 row| / 448 (1 for
 * a zero row) and q = e4m3(bf16 value / s), the decisions of
 * mmdit_quantize_f8 on the bf16 rows; y (device bf16 [B, rows, D]) may be
 * NULL, else the bf16 rows are stored too.  Same shape and alignment rules
 * as mmdit_ln_modulate; errors as there. */
int mmdit_ln_modulate_f8(const float* x, int B, int rows, int D, const float* shift, const float* scale,
                         int64_t mod_stride, float eps, void* y, uint8_t* q, float* s, void* stream);

/* y[b, n] = W act(x[b, :]) + bias, x device fp32 [B, K] (1 <= B <= 16,
 * K <= 6400), act 0 = identity, 1 = SiLU; y device fp32 [B, N].  Rows of x
 * go through the weights 8 at a time. */
int mmdit_gemv(const mmdit_linear_t* lin, int B, int N, int K, const float* x, int act, float* y, void* stream);

/* vec = time2(SiLU(time1(sinusoid(1000 sigma)))) for all B samples:
 * device fp32 [B, D]; ws: device fp32 scratch of B*(t_dim + D) floats. */
int mmdit_time_embed(const mmdit_shape_t* shape, const mmdit_linear_t* time1, const mmdit_linear_t* time2,
                     double sigma, float* vec, float* ws, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MMDIT_H_ */
