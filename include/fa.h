/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact attention forward library.
 *
 * The operation is the exact attention forward pass with its per-row
 * log-sum-exp:
 *
 *     S = scale * Q K^T,   P = softmax(S) (row-wise),   O = P V,
 *     L_i = log sum_j exp(S_ij)
 *
 * ("Flash Attention 4 on Blackwell" (GPU-HPC book, ch. 13), section
 * "Attention's real bottleneck": O = softmax(QK^T / sqrt(d)) V;
 * "Infra: Flash Attention", Algorithm 1 (FlashAttention forward): outputs O and
 * L_i = m_i + log l_i, and section "Why backward recomputes":
 * L_i = log sum_j e^{S_ij}.)
 *
 * The score matrix is never materialised: K/V are streamed in 128-key blocks
 * with an online softmax and conditional rescaling (threshold tau in log2
 * units, "Flash Attention 4 on Blackwell", section "Online softmax and
 * conditional rescaling").
 *
 * Layouts (dense, contiguous, BSHD as in the pages' usage example, section
 * "Build and validation constraints"):
 *   q   [batch, seqlen_q, heads_q,  d_qk]  bf16
 *   k   [batch, seqlen_k, heads_kv, d_qk]  bf16
 *   v   [batch, seqlen_k, heads_kv, d_v ]  bf16
 *   o   [batch, seqlen_q, heads_q,  d_v ]  bf16 (written)
 *   lse [batch, heads_q,  seqlen_q]        fp32, natural log (written; may be NULL)
 * Query head h reads key/value head h / (heads_q / heads_kv) (GQA/MQA,
 * "Flash Attention 4 on Blackwell", section "Causal attention and GQA").
 *
 * Mask: causal = 0 attends to every key.  causal = 1 is the bottom-right
 * aligned mask: query i sees key j iff j <= i + seqlen_k - seqlen_q (same
 * section).  A query row that sees no key (seqlen_q > seqlen_k) gets O = 0
 * and lse = -inf; the pages leave that row to the operator ("Infra: Flash
 * Attention", section "Notation and boundary conditions").
 *
 * Ownership: every tensor pointer is caller-owned device memory on the
 * current CUDA device, 16-byte aligned (TMA requirement).  The library
 * allocates no memory for the caller; it keeps a per-device cache of device
 * properties and a 16-byte device status word.
 *
 * Set-up: the first call of any entry point on a device looks up the
 * library's device arrays, clears the status word and the no-alloc scratch
 * header, and synchronises the device once so that those clears cannot land
 * after later work on a caller's stream.  Make that first call before any
 * stream capture.
 *
 * Ordering: calls are asynchronous and stream-ordered on `stream`; no host
 * synchronisation happens inside.  Argument errors are reported before any
 * CUDA call.  A device-side timeout of the kernel's bounded waits is recorded
 * in the status word and read with fa_device_status().
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers (same underlying type). */
struct CUstream_st;
typedef struct CUstream_st* fa_stream_t;

enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,     /* null pointer, negative size, heads_q % heads_kv != 0, misaligned
                                 or non-device pointer, bad scale or option */
  FA_ERR_UNSUPPORTED = 2,     /* head dims outside {(64,64), (128,64), (128,128), (192,64), (192,128)},
                                 or a device that is not sm_103 / sm_100 family */
  FA_ERR_CUDA = 3,            /* a CUDA runtime/driver call failed (cudaGetLastError is left set) */
  FA_ERR_DEVICE_TIMEOUT = 4,  /* a bounded device wait expired (from fa_device_status) */
  FA_ERR_DEVICE_CHECK = 5     /* a device-side check of the checking build failed (from
                                 fa_device_status; fa_options.debug_flags bit 2) */
};

/*
 * Exact attention forward.
 *
 * batch, heads_q, heads_kv, seqlen_q, seqlen_k >= 0 (heads >= 1 unless batch or
 * seqlen_q is 0); heads_q % heads_kv == 0.  d_qk in {64, 128, 192},
 * d_v in {64, 128}, d_v <= d_qk.  scale multiplies QK^T before the softmax;
 * scale == 0 selects 1/sqrt(d_qk); a negative or non-finite scale is rejected.
 * A problem with batch, heads or seqlen_q equal to 0 returns FA_OK without a
 * launch.  seqlen_k == 0 writes O = 0 and lse = -inf.
 *
 * Returns FA_OK when the work was enqueued.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int batch, int heads_q,
           int heads_kv, int seqlen_q, int seqlen_k, int d_qk, int d_v, int causal, float scale,
           fa_stream_t stream);

/* Options for ablations and tests (fa_fwd uses the defaults). */
typedef struct fa_options {
  float tau;          /* conditional-rescale threshold, log2 units; < 0 selects 8; at most 64,
                         since unnormalised weights reach 2^tau */
  int pack;           /* query heads packed into one 128-row tile; 0 = automatic (the GQA
                         ratio when it divides 128, else 1); otherwise must divide both */
  int grid;           /* persistent CTAs; 0 = one per SM */
  double timeout_s;   /* limit of every device-side wait; <= 0 selects 1 s */
  int debug_flags;    /* bit 0: the softmax warps never signal P ready, so the MMA warp's
                         bounded wait expires (tests the failure path; the output is not
                         valid).  Bit 1 (forward calls): count, per warp of 32 rows and K/V
                         block after the first, the correction warps' rescales of O (the
                         TMEM round trip run when some row of the warp moved its reference
                         by more than tau); read with fa_debug_rescale_count().  Needs
                         exp_emu = 1 or bit 2 (the counter lives in the FMA-exp2 ablation
                         kernel and in the checking build, whose arithmetic is the default
                         kernel's, so the default kernels carry no counting code; the rescale
                         decisions do not depend on how the exponentials are computed), else
                         FA_ERR_UNSUPPORTED.  The output is unchanged.
                         Bit 2 (fixed-length forward with static assignment, no exp_emu):
                         run the checking build of the kernel, which checks every decoded
                         task, TMA tile coordinate, TMEM base and lane quadrant, shared-
                         memory extent and output index before use and, at exit, that each
                         hand-off between the roles was produced as often as it was
                         consumed.  A failed check skips the access, aborts the CTA and
                         records FA_ERR_DEVICE_CHECK with its site (701-707 for the range
                         checks, 710 + i for the hand-off counts) in the status word; the
                         output is then not valid.  The output of a clean run is identical
                         to the default kernel's.  Bit 3 (with bit 2 only): plant a fault
                         for the checks to catch: task 0 decodes to batch index = batch.
                         Other bits must be 0. */
  int exp_emu;        /* 1: compute one in four exponentials of unmasked blocks on the FMA
                         pipe with a degree-3 polynomial instead of the MUFU ex2 unit
                         ("FlashAttention-4 wiki", "Core methods": partial exp emulation);
                         0 (default): MUFU only.  Any other value is rejected. */
  void* workspace;    /* fixed-length calls: NULL (default) assigns tasks to the persistent
                         CTAs round-robin; a device buffer of FA_SCHED_WORKSPACE_BYTES,
                         16-byte aligned, assigns them dynamically (each CTA takes the next
                         task from a counter in it, which the call clears on the stream first;
                         the pages' persistent scheduler with a task counter, "Flash Attention
                         4 on Blackwell", "Scheduling").  Calls that may overlap on different
                         streams need different buffers.  Not combinable with exp_emu; must
                         be NULL for the varlen calls (they take their own workspace). */
  int store_mode;     /* fixed-length epilogue: 0 (default) and 2 write O rows straight from
                         registers; 1 stages them in SMEM and writes them by TMA.  Results
                         are identical; only the speed differs.  Other values are rejected.  Ignored by the varlen, split-KV, dynamic
                         and exp_emu paths. */
  int no_balance;     /* fixed-length calls with static assignment: 0 (default) balances the
                         work of the G persistent CTAs (task t on CTA t mod G).  Without the
                         causal mask: with P tasks and r = P mod G (P when P < G), if
                         0 < 2r <= G and there are at least 4 K/V blocks, the last r tasks
                         are replaced by 2r tasks of one tile each whose two stages take the
                         two halves of the key blocks, merged exactly in the epilogue (row
                         max, row sum and O rescaled to the common maximum); O and LSE agree
                         with the unsplit result up to fp32 rounding.  With the causal mask
                         and an even number of m_blocks: heavy and light m_blocks (m and
                         M-1-m, a constant total of key blocks) are paired on one CTA in
                         consecutive waves; the output is bit-identical.  1 keeps the plain
                         order and whole tasks.  Other values are rejected. */
  uint64_t* trace;    /* NULL (default), or the event log of a fixed-length forward with
                         static assignment, head dims (128, 128) or (192, 128) and no
                         exp_emu or debug bit 2 (else FA_ERR_UNSUPPORTED): device memory of
                         trace_ctas * 5 * (trace_cap + 1) 64-bit words, 8-byte aligned.
                         CTA c < trace_ctas writes five tracks (softmax stage 0, softmax
                         stage 1, correction, MMA, TMA) at word (c * 5 + track) *
                         (trace_cap + 1): the record count, then up to trace_cap records
                         {event code in bits 56-63, argument in bits 32-55, SM clock low
                         32 bits}, stamped by lane 0 of the role's first warp at each step
                         of the hand-off protocol: the waits and arrivals of each role (codes
                         in csrc/fa_kernel.cuh).  A separate kernel build; the output is
                         identical to the default kernel's.  fa_bwd_ex takes it too (head
                         dims (128, 128)): twice the words, the dK/dV kernel's log first,
                         then the dQ kernel's, each with the tracks row warps of stage 0,
                         row warps of stage 1, (unused), MMA, TMA. */
  int trace_ctas;     /* CTAs that record (>= 1 when trace is set) */
  int trace_cap;      /* records kept per track (>= 1 when trace is set) */
  int stagger;        /* 1: an ablation build in which the two softmax warpgroups take turns
                         for their exponentials in the K/V blocks both Q tiles visit (stage 1
                         after stage 0's of the same block, stage 0 after stage 1's of the
                         previous one: the staggered exp sections of "FlashAttention-4 wiki",
                         "Core methods"); fixed-length forward with static assignment, head
                         dims (128, 128) or (192, 128), not with trace, exp_emu or debug bit 2
                         (else FA_ERR_UNSUPPORTED).  The output is identical to the default
                         kernel's.  0 (default): no stagger.  Other values are rejected. */
} fa_options;

#define FA_SCHED_WORKSPACE_BYTES 16

/* Fill `opts` with the defaults. */
void fa_options_default(fa_options* opts);

/* fa_fwd with options; opts == NULL means defaults. */
int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int batch, int heads_q,
              int heads_kv, int seqlen_q, int seqlen_k, int d_qk, int d_v, int causal, float scale,
              const fa_options* opts, fa_stream_t stream);

/*
 * Split-KV forward for decode and other short-query problems.  When the
 * (batch, head group, 256-query block) tasks are too few to fill the GPU, the
 * kernel is starved of parallel work and bound by latency ("FlashAttention-4
 * wiki", "Stress-testing assumptions": the decode failure mode).  Here the
 * keys of every task are cut into `splits` ranges computed by separate CTAs;
 * each writes O / row_sum and its LSE in fp32 to the workspace, and a merge
 * kernel combines them exactly ("Infra: Flash Attention", "Prefill and
 * decode": the merge of softmax states does not fix the scan order, so the
 * keys can be split and merged afterwards; floating-point results differ from
 * fa_fwd only by rounding).
 *
 * Arguments, layouts, masks and results as for fa_fwd_ex, plus:
 *   num_splits  >= 1: key ranges per task (reduced so that none is empty; 1
 *               runs fa_fwd's kernel and ignores the workspace); 0: the
 *               library's choice, fa_splitkv_num_splits() with this device's
 *               SM count.  At most 1024.
 *   workspace   device memory, 16-byte aligned, at least
 *               fa_splitkv_workspace_size(batch, heads_q, seqlen_q, d_v, splits)
 *               bytes for the split count used (partial O [splits, B, Sq, Hq, d_v]
 *               then partial LSE [splits, B, Hq, Sq], fp32); may be NULL when
 *               that count is 1.  Calls that may overlap need different
 *               workspaces.
 * fa_options.workspace and exp_emu must be unset (FA_ERR_UNSUPPORTED).
 * Two launches per call when splitting: the attention kernel and the merge.
 */
int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int batch, int heads_q,
                   int heads_kv, int seqlen_q, int seqlen_k, int d_qk, int d_v, int causal, float scale,
                   int num_splits, void* workspace, size_t workspace_bytes, fa_stream_t stream);

int fa_fwd_splitkv_ex(const void* q, const void* k, const void* v, void* o, float* lse, int batch, int heads_q,
                      int heads_kv, int seqlen_q, int seqlen_k, int d_qk, int d_v, int causal, float scale,
                      int num_splits, void* workspace, size_t workspace_bytes, const fa_options* opts,
                      fa_stream_t stream);

/* Bytes of the split-KV workspace for `num_splits` ranges (0 when num_splits is 1). */
size_t fa_splitkv_workspace_size(int batch, int heads_q, int seqlen_q, int d_v, int num_splits);

/*
 * The split count fa_fwd_splitkv uses for num_splits = 0 on a GPU with
 * num_sms SMs (host only): 1 when the unsplit tasks fill the SMs or the keys
 * are fewer than 8 blocks; otherwise the count (at most 128, at least 4
 * blocks per range, none empty) that minimises waves x (blocks per range + 5):
 * each range pays a start-up of about five block times besides its blocks
 * (fitted to GB300 timings of decode workloads; the smallest such count on a
 * tie).  pack as in fa_options.
 */
int fa_splitkv_num_splits(int batch, int heads_q, int heads_kv, int seqlen_q, int seqlen_k, int d_qk, int d_v,
                          int causal, int pack, int num_sms);

/*
 * Exact attention backward: dQ, dK, dV for a given dO = dLoss/dO, from the
 * forward's inputs, output O and lse ("Infra: Flash Attention", section "Why
 * backward recomputes": P is recomputed from lse, never stored;
 * dV = P^T dO, dP = dO V^T, dS = P (dP - D) with D_i = dO_i . O_i,
 * dQ = scale dS K, dK = scale dS^T Q).  A shared key/value head (GQA/MQA)
 * receives the sum over its query heads.
 *
 * Layouts as fa_fwd: q, dq [batch, seqlen_q, heads_q, d_qk]; o, dout
 * [batch, seqlen_q, heads_q, d_v]; k, dk [batch, seqlen_k, heads_kv, d_qk];
 * v, dv [batch, seqlen_k, heads_kv, d_v]; lse [batch, heads_q, seqlen_q] fp32
 * as fa_fwd writes it.  (d_qk, d_v) in {(64, 64), (128, 128), (192, 128)}
 * (FA_ERR_UNSUPPORTED otherwise).  dq, dk, dv are written whole (bf16).
 *
 * workspace: device memory, 16-byte aligned, at least
 * fa_bwd_workspace_size(batch, heads_q, seqlen_q) bytes: D and lse * log2(e) per query row, padded to
 * whole 128-row blocks.  Calls that may overlap need different workspaces.
 *
 * Three launches on `stream`: the row preparation, the dK/dV kernel and the
 * dQ kernel; no atomics, so the result is deterministic.  seqlen_q == 0
 * writes dK = dV = 0; seqlen_k == 0 writes dQ = 0.  fa_options: grid,
 * timeout_s and debug_flags (bit 0: the row warps never signal P ready, so a
 * bounded wait expires and fa_device_status reports FA_ERR_DEVICE_TIMEOUT)
 * apply, and trace (head dims (128, 128): the event-log build of both
 * kernels, see fa_options.trace); pack > 1, exp_emu, workspace and stagger
 * do not (FA_ERR_UNSUPPORTED when set).
 */
size_t fa_bwd_workspace_size(int batch, int heads_q, int seqlen_q);

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
           void* dq, void* dk, void* dv, int batch, int heads_q, int heads_kv, int seqlen_q, int seqlen_k,
           int d_qk, int d_v, int causal, float scale, void* workspace, size_t workspace_bytes,
           fa_stream_t stream);

int fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
              void* dq, void* dk, void* dv, int batch, int heads_q, int heads_kv, int seqlen_q, int seqlen_k,
              int d_qk, int d_v, int causal, float scale, void* workspace, size_t workspace_bytes,
              const fa_options* opts, fa_stream_t stream);

/*
 * Backward of a variable-length batch: dQ, dK, dV of fa_fwd_varlen's output
 * ("Infra: Flash Attention", section "Why backward recomputes", applied to
 * each sequence as its own problem).  Layouts as fa_fwd_varlen's: q, dq
 * [total_q, heads_q, d_qk]; k, dk [total_k, heads_kv, d_qk]; v, dv
 * [total_k, heads_kv, d_v]; o, dout [total_q, heads_q, d_v] bf16; lse
 * [heads_q, total_q] fp32 (the forward's); cu_seqlens_q / cu_seqlens_k int32
 * [batch + 1] in device memory (sequence b: query rows cu_seqlens_q[b] ..
 * cu_seqlens_q[b+1]-1, key rows likewise; causal is bottom-right inside each
 * sequence).  Head dims (64, 64), (128, 128), (192, 128); batch <= 8192.
 * Rows outside every sequence are neither read nor written, except that
 * total_q == 0 zeroes the whole of dk and dv and total_k == 0 the whole of
 * dq.  A sequence without queries gets dK = dV = 0, one without keys dQ = 0.
 *
 * workspace: device memory of fa_bwd_varlen_workspace_size(batch, heads_q,
 * heads_kv, total_q, total_k) bytes, 16-byte aligned (the planned task lists
 * and D, LSE * log2(e) per padded query row); calls that may overlap need
 * different workspaces.  Stream-ordered launches: a planning kernel (one
 * CTA: checks cu_seqlens, orders the sequences longest first and writes the
 * task records), the row preparation, the dK/dV kernel and the dQ kernel;
 * deterministic.  Bad cu_seqlens: nothing is computed and fa_device_status
 * reports FA_ERR_INVALID_ARG with site 501 and the sequence index.
 * fa_options: grid, timeout_s and debug_flags bit 0 apply; pack > 1,
 * exp_emu, workspace, trace and stagger are FA_ERR_UNSUPPORTED.
 */
size_t fa_bwd_varlen_workspace_size(int batch, int heads_q, int heads_kv, int64_t total_q, int64_t total_k);

int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                  void* dq, void* dk, void* dv, const int* cu_seqlens_q, const int* cu_seqlens_k, int batch,
                  int64_t total_q, int64_t total_k, int heads_q, int heads_kv, int d_qk, int d_v, int causal,
                  float scale, void* workspace, size_t workspace_bytes, fa_stream_t stream);

int fa_bwd_varlen_ex(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, const int* cu_seqlens_q, const int* cu_seqlens_k, int batch,
                     int64_t total_q, int64_t total_k, int heads_q, int heads_kv, int d_qk, int d_v, int causal,
                     float scale, void* workspace, size_t workspace_bytes, const fa_options* opts,
                     fa_stream_t stream);

/*
 * Test hook for the emulated exponential: for i < n, y_fma[i] = 2^x[i] by the
 * FMA-pipe polynomial used with exp_emu = 1, y_mufu[i] = the hardware ex2
 * (ex2.approx.ftz).  Device pointers, fp32; stream-ordered.
 */
int fa_selftest_exp2(const float* x, float* y_fma, float* y_mufu, int n, fa_stream_t stream);

/*
 * Variable-length batches: `batch` sequences of different lengths packed back
 * to back ("FlashAttention-4 wiki", "Core methods" and "Limitations": varlen
 * is supported, with a preprocessing kernel that orders the batch longest
 * first).  Sequence b holds queries cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and
 * keys cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1; each sequence is an independent
 * attention problem with the same heads, head dims, scale and mask rule as
 * fa_fwd (causal = bottom-right inside each sequence).
 *
 * Layouts (dense, contiguous):
 *   q   [total_q, heads_q,  d_qk]  bf16
 *   k   [total_k, heads_kv, d_qk]  bf16
 *   v   [total_k, heads_kv, d_v ]  bf16
 *   o   [total_q, heads_q,  d_v ]  bf16 (rows of the sequences written; other rows untouched)
 *   lse [heads_q, total_q]         fp32, natural log (may be NULL)
 *   cu_seqlens_q, cu_seqlens_k     int32 [batch + 1], device memory
 * The offsets must satisfy 0 <= cu[b] <= cu[b+1] <= total.  They live on the
 * device, so they are checked there: on a violation nothing is computed and
 * the status word (fa_device_status) reports FA_ERR_INVALID_ARG with site 501
 * and the first bad sequence index.  q rows past the end of a sequence may be
 * read (and ignored), never written.
 *
 * workspace: caller-owned device memory, 16-byte aligned, at least
 * fa_varlen_workspace_size(batch, heads_q, total_q) bytes.  Each call writes
 * its task list there (an int task count at byte 0, fa_varlen_task records
 * from byte 256) with a one-block planning kernel and the attention kernel
 * reads it, both on `stream`; calls ordered on one stream may share a
 * workspace, concurrent calls may not.
 *
 * batch <= 16384; total_q + total_k < 2^31 - 512.  total_k == 0 writes O = 0
 * and lse = -inf for every query row.  fa_options.exp_emu must be 0
 * (FA_ERR_UNSUPPORTED otherwise).  Other arguments as for fa_fwd_ex.
 */
typedef struct fa_varlen_task {
  int b, g, mblock, reserved;   /* sequence, head group, m_block (as fa_task) */
  int q_row0, seqlen_q;         /* cu_seqlens_q[b], its query count */
  int k_row0, seqlen_k;         /* cu_seqlens_k[b], its key count */
} fa_varlen_task;

size_t fa_varlen_workspace_size(int batch, int heads_q, int64_t total_q);

int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, int batch, int64_t total_q, int64_t total_k, int heads_q,
                  int heads_kv, int d_qk, int d_v, int causal, float scale, void* workspace,
                  size_t workspace_bytes, fa_stream_t stream);

int fa_fwd_varlen_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                     const int* cu_seqlens_q, const int* cu_seqlens_k, int batch, int64_t total_q,
                     int64_t total_k, int heads_q, int heads_kv, int d_qk, int d_v, int causal, float scale,
                     void* workspace, size_t workspace_bytes, const fa_options* opts, fa_stream_t stream);

/*
 * fa_fwd_varlen without a caller workspace: the planning workspace lives in a
 * file-scope device array of the library (fa_noalloc_scratch_bytes() bytes,
 * 1 MiB, one per device; its address is looked up once per device at set-up).
 * The pages have no counterpart: this is a convenience of this library for
 * callers that cannot hand it scratch memory, such as runtimes that own all
 * device memory through a fixed arena or pool and give a kernel library only
 * its input and output tensors, or code that must not call cudaMalloc (which
 * may synchronise the device) on its serving path.  Nothing is allocated: no
 * cudaMalloc, cudaFree or allocating library routine is called.  The first
 * call on a device does the one-time set-up described at the top of this
 * file (the array's address, its header cleared), so make it before any
 * stream capture.
 *
 * A call whose task list needs more than the array holds
 * (fa_varlen_workspace_size(batch, heads_q, total_q) > 1 MiB, about 32 760
 * tasks) is rejected with FA_ERR_INVALID_ARG before any CUDA call.  Other
 * arguments, errors and outputs as for fa_fwd_varlen.
 *
 * Race: every call on a device shares the one array.  Two calls that overlap
 * in time (different streams without ordering between them, or host threads
 * issuing concurrently to different streams) overwrite each other's task
 * list and task counter, and their outputs are then undefined.  Calls
 * ordered on one stream are safe; otherwise order them (events or
 * synchronisation) or use fa_fwd_varlen with one workspace per stream.
 */
int fa_fwd_varlen_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                          const int* cu_seqlens_q, const int* cu_seqlens_k, int batch, int64_t total_q,
                          int64_t total_k, int heads_q, int heads_kv, int d_qk, int d_v, int causal,
                          float scale, fa_stream_t stream);

/* Bytes of the static scratch array used by fa_fwd_varlen_noalloc. */
size_t fa_noalloc_scratch_bytes(void);

/*
 * Host-only copy of the planning kernel's task list (no CUDA call): the same
 * records in the same order, for host cu_seqlens arrays.  l2_bytes is the L2
 * budget of the causal sections (0 selects 64 MiB; the kernel uses half the
 * device's L2).  Writes min(count, capacity) records to `out` (may be NULL)
 * and the task count to *count.
 */
int fa_varlen_plan_host(const int* cu_seqlens_q, const int* cu_seqlens_k, int batch, int heads_q, int heads_kv,
                        int d_qk, int d_v, int causal, int64_t l2_bytes, int pack, fa_varlen_task* out,
                        int64_t capacity, int64_t* count);

/*
 * Synchronise `stream`, then read and clear the current device's status
 * word.  *out receives FA_OK, FA_ERR_DEVICE_TIMEOUT, FA_ERR_DEVICE_CHECK (a
 * check of the checking build failed) or FA_ERR_INVALID_ARG (a varlen call
 * found bad cu_seqlens).  Returns FA_OK or FA_ERR_CUDA.
 */
int fa_device_status(fa_stream_t stream, int* out);

/*
 * The same, with the recorded detail: detail (may be NULL) receives {code,
 * site, block or sequence index}, the site being the wait or check that
 * failed: 101-404 a forward wait (role * 100 + barrier: 1 softmax,
 * 2 correction, 3 MMA, 4 TMA), 501 bad cu_seqlens, 502 a varlen batch with
 * more tasks than the workspace holds, 601-623 a backward wait,
 * 701-707 a range check and 710 + i a hand-off count of the checking build.
 */
int fa_device_status_detail(fa_stream_t stream, int* out, unsigned int detail[3]);

/*
 * Synchronise `stream`, then read and clear the current device's counter of
 * O rescales (forward calls made with fa_options.debug_flags bit 1; the
 * counter is also cleared by fa_device_status).  Returns FA_OK or FA_ERR_CUDA.
 */
int fa_debug_rescale_count(fa_stream_t stream, unsigned int* out);

/* Human-readable name of a status code (static storage). */
const char* fa_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int fa_version(void);

/*
 * Host-only view of the tile decomposition the kernel runs (no CUDA call).
 * A task is (batch b, head group g, m_block): two consecutive 128-row Q tiles
 * ("stages") that stream the same K/V blocks ("Flash Attention 4 on
 * Blackwell", section "Scheduling": tasks (batch, kv_head, m_block), each
 * m_block holding two Q stages; causal tasks run longest first).  Causal
 * order: the heavier half of the m_blocks in L2 sections (decreasing m inside
 * a section), then the lighter half one m_block level at a time.
 */
typedef struct fa_plan {
  int batch, heads_q, heads_kv, seqlen_q, seqlen_k, causal;
  int pack;            /* query heads per tile */
  int groups;          /* heads_q / pack */
  int pos_per_tile;    /* 128 / pack sequence positions per tile */
  int tiles;           /* Q tiles per (b, g) */
  int mblocks;         /* tasks per (b, g) */
  int kv_blocks;       /* ceil(seqlen_k / 128) */
  int ratio;           /* heads_q / heads_kv */
  int section_units;   /* causal order: (b, g) units per L2 section */
  int heavy_levels;    /* causal order: the top heavy_levels m_blocks go section by section,
                          the rest level by level over all units */
  int64_t num_tasks;
  int64_t tail_first;  /* first key-split task of a balanced last wave (= num_tasks: none) */
  int grid;            /* 0: the plain order; else the balanced static order for this many
                          CTAs (set by fa_plan_set_grid) */
} fa_plan;

typedef struct fa_task {
  int b, g, mblock, kv_head;
  int pos0[2];         /* first sequence position of each stage's tile */
  int n_blocks[2];     /* K/V blocks each stage visits */
  int key_split;       /* key-split task: both stages hold the tile at pos0[0]; stage 0 visits
                          key blocks [0, key_split), stage 1 the next n_blocks[1]; else 0 */
} fa_task;

/* l2_bytes: K/V bytes per section of the causal order (0 selects 8 MiB: what
   fa_fwd uses, min(L2 size / 2, 8 MiB), on an L2 of 16 MiB or more). */
int fa_make_plan(int batch, int heads_q, int heads_kv, int seqlen_q, int seqlen_k, int d_qk, int d_v,
                 int causal, int64_t l2_bytes, int pack, fa_plan* out);
int fa_plan_task(const fa_plan* plan, int64_t task, fa_task* out);

/* The balanced static order fa_fwd runs on `grid` persistent CTAs (the SM count
   by default; see fa_options.no_balance): sets plan->grid and updates num_tasks
   and tail_first of a plan made by fa_make_plan (FA_ERR_INVALID_ARG if already
   applied or grid < 1).  fa_plan_task then returns the tasks in that order
   (empty entries of the paired causal order have n_blocks = {0, 0} and
   pos0 = {seqlen_q, seqlen_q}).  Plans that gain nothing are left unchanged. */
int fa_plan_set_grid(fa_plan* plan, int grid);

/* Does block j need the element mask for a tile starting at pos0? (host view) */
int fa_plan_block_masked(const fa_plan* plan, int pos0, int j);

/* The first block that needs it; the kernel masks exactly the blocks j >= this
   index (the tail and the causal diagonal only grow with j). */
int fa_plan_first_masked_block(const fa_plan* plan, int pos0);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
