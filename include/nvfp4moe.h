/*
 * nvfp4moe.h -- C ABI of the GB300 (sm_103a) NVFP4 decode library.
 *
 * The library computes the decode-time "skinny" matmuls of 4-bit NVFP4
 * models: 1..32 rows of BF16 activations times a large NVFP4 weight matrix
 * (W4A16), as a dense projection / head (with an optional fused argmax) and as
 * a top-k routed mixture-of-experts layer with an always-on shared expert.
 *
 * Sources.  "Qwen3.6-35B-A3B NVFP4 on an RTX 5090 (Elsa)", section "Making
 * decode faster": paragraph "Skinny matrix multiplies" (decode matmuls are
 * four to sixteen rows of 16-bit activations times a large weight matrix,
 * 4-bit weights with 16-bit activations; split-K), paragraph "One environment
 * variable" (the fused MoE finalize: weighted top-k combine), paragraph
 * "FR-Spec, and a silent bug" (a 4-bit head).  The pages name NVFP4 without
 * defining it; the layout below is this library's specification of it.
 *
 * NVFP4 layout (plain row-major, no repacking):
 *   codes  uint8 [N, K/2]   E2M1 codes, byte j of a row holds k = 2j in bits
 *                           3..0 and k = 2j+1 in bits 7..4;
 *   scales uint8 [N, K/16]  FP8 E4M3 ("fn") scale of the block k / 16;
 *   global float32 (device) per-tensor scale;
 *   W[n][k] = e2m1(code) * e4m3(scale) * global.
 *
 * Conventions for every entry point:
 *   - All pointers are DEVICE pointers unless stated otherwise.  The caller
 *     owns every buffer; the library never allocates, frees or synchronises
 *     in a compute call.  Calls are asynchronous on `stream` and may be
 *     captured in a CUDA graph.
 *   - Activations are BF16 (uint16 bit patterns of bfloat16), row-major with
 *     a leading dimension in elements.  Pointers and leading dimensions must
 *     give 16-byte aligned rows; weight pointers must be 16-byte aligned.
 *   - Dense NVFP4 calls take K % 32 == 0 (two E4M3 scale bytes per row per
 *     32 K); everything else streams 256-K stages and takes K, H, I % 256 ==
 *     0 (the scales' row pitch K / 16 must then be a multiple of 16 bytes,
 *     which tensor-memory-access copies need).  1 <= M, T <= 32.
 *   - Return value: NVFP4_OK or a negative status.  On a negative status
 *     nothing was launched and nvfp4_last_error() describes why.  No C++
 *     exception crosses this boundary.
 *   - Workspace: a device buffer of at least the queried size, zero-filled
 *     once before its first use (nvfp4_workspace_init).  Every call keeps
 *     the same header (status word, then tile counters that kernels leave at
 *     zero again) and puts its scratch after it, so one workspace of the
 *     largest queried size may serve any sequence of calls on one stream.
 *     It must not be used by two calls that may run concurrently.
 *   - Problems found on the device (an expert id outside [0, E), a pipeline
 *     wait that gave up) never trap: they set bits in the workspace's status
 *     word, read by nvfp4_read_device_status().
 */
#ifndef NVFP4MOE_H
#define NVFP4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (same type); NULL is the legacy default stream. */
typedef struct CUstream_st* nvfp4_stream_t;

enum {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID = -1,   /* null pointer, bad count, k > E ... */
  NVFP4_ERR_ALIGN = -2,     /* pointer / leading dimension not 16-byte aligned */
  NVFP4_ERR_SHAPE = -3,     /* K not a supported multiple, M or T outside [1, 32], E too large */
  NVFP4_ERR_ARCH = -4,      /* current device is not compute capability 10.3 */
  NVFP4_ERR_CUDA = -5,      /* a CUDA runtime / launch error */
  NVFP4_ERR_WORKSPACE = -6  /* workspace missing or smaller than required */
};

/* call flags */
#define NVFP4_FLAG_RMS_INPUT 1u /* scale each input row by 1/sqrt(mean(x^2)+1e-6) */
/* Launch without programmatic dependent launch.  With it (the default) a
 * call's kernels may start while the previous kernel on the stream runs, and
 * read their weights (codes, scales, global scales: never outputs of the
 * previous kernel) before waiting for it; activations (and routing ids and
 * weights, unless NVFP4_FLAG_IDS_READY) are read after the wait.  A caller
 * whose previous kernel writes a weight and lets its dependents start early
 * passes this flag. */
#define NVFP4_FLAG_NO_PDL 2u
/* moe_nvfp4_decode: the ids and weights were complete before the previous
 * kernel on the stream started (e.g. routing done earlier in the step), so
 * the kernels may read them, and start streaming the routed experts'
 * weights, before waiting for that kernel to finish. */
#define NVFP4_FLAG_IDS_READY 4u
/* Program ops (nvfp4_program_create) only: split this op over the CTAs
 * exactly as its single call does on the tensor cores (every SM, or for a
 * dense op with fewer 128-row tiles than SMs, tiles x ceil(K / 1024) CTAs),
 * so its results are bit-identical to that call's (a single call that its
 * shape sends to the CUDA-core kernels adds in another order).  Without it
 * a small NVFP4 dense op of a program runs on tiles x ceil(K / 2048) CTAs
 * (whole 128-row tiles or few K splits each) while the other SMs stream the
 * next ops' weights. */
#define NVFP4_FLAG_ALL_SMS 8u

/* device status bits */
#define NVFP4_STATUS_BAD_EXPERT_ID 1u /* an id outside [0, E): its slot was skipped */
#define NVFP4_STATUS_WAIT_TIMEOUT 2u  /* a pipeline wait gave up; outputs invalid */

typedef struct nvfp4_weight {
  const uint8_t* codes;       /* [n, k/2] */
  const uint8_t* scales;      /* [n, k/16] */
  const float* global_scale;  /* 1 float */
  int32_t n, k;
} nvfp4_weight;

/* E experts stacked: gu_codes [E, 2I, H/2], gu_scales [E, 2I, H/16],
 * dn_codes [E, H, I/2], dn_scales [E, H, I/16], gu_global / dn_global [E].
 * Rows [0, I) of each gate_up matrix are the gate, rows [I, 2I) the up
 * projection.  A single (shared) expert is a stack with E = 1. */
typedef struct nvfp4_expert_stack {
  const uint8_t* gu_codes;
  const uint8_t* gu_scales;
  const uint8_t* dn_codes;
  const uint8_t* dn_scales;
  const float* gu_global;
  const float* dn_global;
  int32_t num_experts, hidden, inter;
} nvfp4_expert_stack;

/* NVFP4_OK if `device` is compute capability 10.3 (GB300), else
 * NVFP4_ERR_ARCH (or NVFP4_ERR_CUDA if the device cannot be queried). */
int nvfp4_device_check(int device);

/* Zero-fill a workspace (asynchronous, on `stream`). */
int nvfp4_workspace_init(void* workspace, size_t bytes, nvfp4_stream_t stream);

/* ---- dense skinny GEMM --------------------------------------------------
 * C[m][n] = bf16( sum_k A'[m][k] * W[n][k] ),  m < M, n < W->n,
 * accumulated in FP32 after each activation row is brought to FP16 exactly
 * by a power-of-two scale; A' = A, or with NVFP4_FLAG_RMS_INPUT
 * A'[m] = A[m] / sqrt(mean_k A[m][k]^2 + 1e-6) (FP32).
 *   A [M, lda] bf16, lda >= K;  C [M, ldc] bf16, ldc >= N.
 *   argmax_out: NULL, or int32 [M]: index of the first maximum of each row of
 *   the BF16 output C (ties to the lowest index).
 * Split-K partial sums are reduced in a fixed order: results are
 * deterministic.  K % 32 == 0.  Two kernels serve it, chosen by shape alone
 * (nvfp4_last_dispatch names the one that ran): the tensor-core kernel
 * streams 256-K stages through tcgen05 MMAs and costs about 13 us a call
 * before its first byte; the CUDA-core kernel (whole rows per warp, FP32
 * accumulation of the same exact FP16 products) starts in a few us but does
 * one FMA per weight and row (more than four rows run as CTAs of four rows
 * in ceil(M / 4) row groups).  The CUDA cores take every K % 256 != 0, and
 * K % 256 == 0 when the weight (codes + scales) is at most 128 MiB for
 * M = 1, 20 MiB for M = 2, 3 and 10 MiB for M = 4; for M = 5..16 when it is
 * at most 5 MiB and ceil(N / 16) * ceil(M / 4) <= 2 x the SM count (one
 * wave of its CTAs).
 * The two differ only in the order of the FP32 additions (a few units in
 * the last place of C). */
size_t nvfp4_gemm_skinny_workspace(int M, int N, int K);
int nvfp4_gemm_skinny(const void* A, int64_t lda, int M, const nvfp4_weight* W,
                      void* C, int64_t ldc, int32_t* argmax_out, uint32_t flags,
                      void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* ---- other weight formats on the same path ------------------------------
 * "Qwen3.6-35B-A3B NVFP4 on an RTX 5090 (Elsa)", section "Making decode
 * faster": paragraph "An FP8 fast path that never ran" (small-batch
 * projections with FP8 weights and one per-tensor weight scale: 0.85 -> 1.4
 * TB/s once the FP8 kernel engaged) and paragraph "Skinny matrix
 * multiplies" (the 2048 -> 64 projections and the 4-bit shared experts
 * expanded to BF16 at load, run by a split-K kernel: 8.7 us -> 2.8 us).
 *
 * fp8_gemm_skinny: W8A16.  codes uint8 [n, k] E4M3 ("fn") bytes, row-major;
 * scale: device pointer to one float32.
 *   C[m][n] = bf16( scale * sum_k A'[m][k] * e4m3(codes[n][k]) ).
 * bf16w_gemm_skinny: BF16 weights w [n, ldw] (k columns used), row-major.
 *   C[m][n] = bf16( sum_k A'[m][k] * w[n][k] ).
 * Everything else as nvfp4_gemm_skinny: A' (NVFP4_FLAG_RMS_INPUT), argmax_out,
 * flags, FP32 accumulation, deterministic split-K, the workspace rules, the
 * status codes.  K % 256 == 0; codes / w 16-byte aligned (ldw % 8 == 0).  The
 * FP8 codes are decoded to FP16 exactly and multiply activation rows staged
 * as FP16 exactly (as for NVFP4); BF16 weights multiply the BF16
 * activations as they are. */
typedef struct fp8_weight {
  const uint8_t* codes;  /* [n, k] */
  const float* scale;    /* 1 float */
  int32_t n, k;
} fp8_weight;

typedef struct bf16_weight {
  const void* w;  /* [n, ldw] bf16 */
  int64_t ldw;
  int32_t n, k;
} bf16_weight;

size_t fp8_gemm_skinny_workspace(int M, int N, int K);
int fp8_gemm_skinny(const void* A, int64_t lda, int M, const fp8_weight* W, void* C, int64_t ldc,
                    int32_t* argmax_out, uint32_t flags, void* workspace, size_t workspace_bytes,
                    nvfp4_stream_t stream);
size_t bf16w_gemm_skinny_workspace(int M, int N, int K);
int bf16w_gemm_skinny(const void* A, int64_t lda, int M, const bf16_weight* W, void* C,
                      int64_t ldc, int32_t* argmax_out, uint32_t flags, void* workspace,
                      size_t workspace_bytes, nvfp4_stream_t stream);

/* ---- dense skinny GEMM without a workspace -------------------------------
 * (This library's own addition; the pages have no counterpart.)  Same
 * arguments and results as nvfp4_gemm_skinny minus the workspace, for
 * callers that cannot allocate device memory (a plugin whose host runtime
 * owns every allocation, a real-time loop that may not call cudaMalloc, a
 * process with a fixed memory budget).  Scratch comes from an 8 MiB array
 * built into the library, held on every GPU that loads it until exit; a
 * shape that needs more is rejected with NVFP4_ERR_WORKSPACE.  The first call
 * on a device (with that device current) looks the array's address up; make
 * it before any stream capture.  The address is kept for the life of the
 * process: resetting the device while the library is loaded is not
 * supported.  Every argument is checked first; a refused call touches
 * nothing.  Each accepted call clears the array's status word and counters on
 * `stream` first.  All calls share the one array: calls that may overlap on
 * the GPU (other streams, concurrent graphs) race and must not be issued. */
int nvfp4_gemm_skinny_noalloc(const void* A, int64_t lda, int M, const nvfp4_weight* W,
                              void* C, int64_t ldc, int32_t* argmax_out, uint32_t flags,
                              nvfp4_stream_t stream);

/* ---- hot-vocabulary head --------------------------------------------------
 * "Qwen3.6-35B-A3B NVFP4 on an RTX 5090 (Elsa)", section "Making decode
 * faster", paragraph "FR-Spec, and a silent bug": the draft scores only a
 * list of the most likely tokens (32K) through a 4-bit head built from the
 * checkpoint's output head (37 MB a draft step instead of the full head).
 *
 * nvfp4_gather_rows builds that head once: codes [n_rows, K/2] and scales
 * [n_rows, K/16] receive rows rows[0..n_rows) of src, in list order (the
 * plain row-major layout keeps each row contiguous, so this is exact; a row
 * id outside [0, src->n) gives an all-zero row).  rows: int32 [n_rows] on
 * the device; codes / scales: caller-owned device arrays, 16-byte aligned,
 * not overlapping src.  K % 256 == 0.  Asynchronous on `stream`.  The hot
 * head's global scale is src's (pass src->global_scale).
 *
 * nvfp4_hot_vocab_head is nvfp4_gemm_skinny on the hot head W_hot
 * [n_hot, K] (C [M, n_hot] = the hot rows' BF16 logits) whose argmax_out
 * (required) reports vocabulary ids: argmax_out[m] = vocab_ids[j], j the
 * first maximum of C[m] (ties to the lowest hot row; with ascending
 * vocab_ids that is the lowest vocabulary id).  vocab_ids: int32 [n_hot] on
 * the device (the list the head was gathered with).  Workspace:
 * nvfp4_gemm_skinny_workspace(M, n_hot, K). */
int nvfp4_gather_rows(const nvfp4_weight* src, const int32_t* rows, int n_rows, void* codes,
                      void* scales, nvfp4_stream_t stream);
int nvfp4_hot_vocab_head(const void* A, int64_t lda, int M, const nvfp4_weight* W_hot,
                         const int32_t* vocab_ids, void* C, int64_t ldc, int32_t* argmax_out,
                         uint32_t flags, void* workspace, size_t workspace_bytes,
                         nvfp4_stream_t stream);

/* ---- BF16 -> NVFP4 quantisation --------------------------------------------
 * "Qwen3.8-27B-NVFP4-lmhead4-recipe" (model card), section "Files": a BF16
 * head converted to NVFP4 (the tool's rule is not given; this is the usual
 * NVFP4 recipe).  W bf16 [N, ldw] row-major (K columns used) ->
 *   global_scale (1 float, device) g = amax|W| / (6 * 448), 1 if W is all 0;
 *   scales [N, K/16]: E4M3 of amax of each 16-element block / (6 g);
 *   codes [N, K/2]: E2M1 of |x| / (e4m3(scale) * g) with x's sign (a code
 *   rounded to 0 is +0), two per byte, low nibble = even k.
 * Roundings to nearest, ties to the even code, saturating at 448 / 6; every
 * quotient and product one float32 operation (deterministic).  The result
 * is a plain nvfp4_weight {codes, scales, global_scale, N, K}.  K % 32 == 0;
 * W rows and codes 16-byte aligned; outputs caller-owned device memory.
 * Asynchronous on `stream` (three kernels; global_scale holds a partial
 * result until the last one ends). */
int nvfp4_quantize(const void* W, int64_t ldw, int N, int K, void* codes, void* scales,
                   float* global_scale, nvfp4_stream_t stream);

/* ---- top-k softmax routing ----------------------------------------------
 * logits float32 [T, E] (row-major).  For each row the k experts with the
 * largest logits, compared as float32, ties to the lower index, listed in
 * that order -> topk_ids int32 [T, k].  topk_w float32 [T, k]: softmax
 * probabilities, renormalised over the chosen k when `renormalize` != 0.
 * Limits: 1 <= k <= E <= 512, k <= 32, T >= 1 (any T: rows are independent). */
int topk_softmax_route(const float* logits, int T, int E, int k, int renormalize,
                       int32_t* topk_ids, float* topk_w, nvfp4_stream_t stream);

/* ---- MoE decode layer ----------------------------------------------------
 * out[t] = bf16( sum_j w[t][j] * E_{ids[t][j]}(x'[t]) + E_shared(x'[t]) ),
 * E(x) = W_down (silu(W_gate x) * (W_up x)), silu(z) = z / (1 + exp(-z)).
 * Only the experts some token routes to are read.  x' as A' above.
 *   x [T, ldx] bf16 (ldx >= H);  topk_ids int32 [T, k];  topk_w float32 [T, k];
 *   experts: the routed stack; shared: NULL or a stack with E = 1 and the
 *   same H and I;  out [T, ldo] bf16.
 * Intermediates (gate/up sums, silu(g)*u, per-expert down outputs and the
 * combine) are FP32; the per-slot outputs are summed in slot order, the
 * shared expert last: deterministic.  Ids outside [0, E) are skipped and set
 * NVFP4_STATUS_BAD_EXPERT_ID.  Limits: T <= 32, k <= 16, E <= 512,
 * H % 256 == 0, I % 256 == 0.  With I in {256, 512, 1024} (and 16 x H x 2
 * bytes within 96 KB) two CUDA-core kernels serve the call, per batch of at
 * most 16 tokens: gate/up + SwiGLU per (token, slot) pair (for batches of 4
 * to 8 tokens with H % 512 == 0 by warp-level MMAs, FP16 x FP16 -> FP32),
 * then down with the combine; the tensor-core kernels (gate_up, down,
 * combine) take the other shapes.  They differ only in the order of FP32
 * additions and in h's FP16 staging (nvfp4_last_dispatch names the
 * kernels). */
size_t moe_nvfp4_decode_workspace(int T, int k, const nvfp4_expert_stack* experts);
int moe_nvfp4_decode(const void* x, int64_t ldx, int T, const int32_t* topk_ids,
                     const float* topk_w, int k, const nvfp4_expert_stack* experts,
                     const nvfp4_expert_stack* shared, void* out, int64_t ldo,
                     uint32_t flags, void* workspace, size_t workspace_bytes,
                     nvfp4_stream_t stream);

/* ---- programs: a chain of calls in one launch -----------------------------
 * (This library's own runtime; the pages run each matmul as its own kernel
 * replayed from a CUDA graph.)  A program is a fixed sequence of GEMM and MoE
 * calls in which each call may read what the calls before it wrote, e.g. the
 * projections and MoE layers of a whole decode step.  nvfp4_program_launch
 * runs the sequence in one cooperative launch with one CTA per SM: each SM
 * keeps streaming the weights of the calls ahead while the current call's
 * split-K reductions finish, and a call reads its activations only once every
 * CTA has finished the call before it (completion counters in the workspace).
 * Each op computes what its single call computes, always on the tensor
 * cores (the tcgen05 kernel's path of that call).  A small dense op may have
 * its K range split over fewer CTAs than the single call would use, which
 * changes the order in which FP32 split-K partials are added, so its output
 * can differ from the single call's in the last bits; every launch of one
 * program gives bit-identical results.
 *
 * nvfp4_op: kind NVFP4_OP_GEMM takes the arguments of nvfp4_gemm_skinny (A,
 * lda, M, W, C, ldc, argmax_out) and, for a hot-vocabulary head, argmax_map
 * (NULL, or vocab_ids as in nvfp4_hot_vocab_head; needs argmax_out), kind
 * NVFP4_OP_MOE those of moe_nvfp4_decode
 * (x ... ldo; shared.num_experts == 0 means no shared expert).  flags:
 * NVFP4_FLAG_RMS_INPUT and NVFP4_FLAG_ALL_SMS per op (NVFP4_FLAG_NO_PDL and
 * NVFP4_FLAG_IDS_READY are accepted and ignored).  Every MoE op's topk_ids / topk_w must be complete
 * before the launch (e.g. routed earlier on the stream).  Limits as for the
 * single calls; at most 4,095 kernel ops (a MoE op counts three: gate_up,
 * down, combine).
 *
 * nvfp4_program_create validates every op, encodes its tensor maps, and
 * copies the op table to device memory: the one call of this library that
 * allocates (cudaMalloc) and synchronises; do it once, before any capture.
 * The program binds every pointer given, including the workspace (at least
 * nvfp4_program_workspace() bytes, zero-filled once); nvfp4_program_launch is
 * asynchronous and graph-capturable.  The workspace must not be used by
 * another call while a launch may be running.  nvfp4_program_destroy frees
 * the table (after the last launch has finished). */
enum { NVFP4_OP_GEMM = 1, NVFP4_OP_MOE = 2 };

typedef struct nvfp4_op {
  int32_t kind;
  uint32_t flags;
  /* NVFP4_OP_GEMM */
  const void* A;
  int64_t lda;
  int32_t M;
  nvfp4_weight W;
  void* C;
  int64_t ldc;
  int32_t* argmax_out;
  /* NVFP4_OP_MOE */
  const void* x;
  int64_t ldx;
  int32_t T;
  const int32_t* topk_ids;
  const float* topk_w;
  int32_t k;
  nvfp4_expert_stack experts;
  nvfp4_expert_stack shared;
  void* out;
  int64_t ldo;
  /* NVFP4_OP_GEMM, hot-vocabulary head */
  const int32_t* argmax_map;
} nvfp4_op;

typedef struct nvfp4_program nvfp4_program;

size_t nvfp4_program_workspace(const nvfp4_op* ops, int n_ops);
int nvfp4_program_create(const nvfp4_op* ops, int n_ops, void* workspace,
                         size_t workspace_bytes, nvfp4_program** program);
int nvfp4_program_launch(const nvfp4_program* program, nvfp4_stream_t stream);
int nvfp4_program_destroy(nvfp4_program* program);

/* ---- diagnostics ---------------------------------------------------------
 * Copy the workspace's status word to *flags and clear it.  Synchronises
 * `stream`: for tests, not for the decode loop. */
int nvfp4_read_device_status(void* workspace, uint32_t* flags, nvfp4_stream_t stream);

/* Measurement aid (this library's own; the pages have none): read `bytes`
 * (a positive multiple of 16) of the device buffer `buf` (16-byte aligned)
 * once, as a plain streaming kernel does (16-byte loads that bypass L1,
 * eight in flight per thread, two CTAs per SM), and write one word per CTA
 * to `sink` (device, at least 8 * SMs bytes) so no load can be dropped.
 * Timing it over a buffer much larger than L2 gives the read-only HBM
 * bandwidth, the second denominator for the weight stream's roofline.
 * Asynchronous on `stream`. */
int nvfp4_hbm_read_probe(const void* buf, size_t bytes, void* sink, size_t sink_bytes,
                         nvfp4_stream_t stream);

/* Text describing the launches of this thread's last successful call
 * (kernel, grid, work items, split): tests assert the intended path ran.
 * Writes at most n bytes including the terminating NUL; returns the length. */
int nvfp4_last_dispatch(char* buf, size_t n);

/* Message for this thread's last failed call ("" if none). */
const char* nvfp4_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4MOE_H */
