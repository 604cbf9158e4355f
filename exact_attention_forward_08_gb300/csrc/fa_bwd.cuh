// Exact attention backward for sm_103a: dQ, dK, dV for a given dO, from the
// forward's O and LSE ("Infra: Flash Attention", section "Why backward
// recomputes" and its detail on the block-wise gradients):
//
//   P = exp(scale * Q K^T - LSE)        (recomputed, never stored)
//   dV = P^T dO          dP = dO V^T
//   dS = P (dP - D),     D_i = dO_i . O_i
//   dQ = scale dS K      dK = scale dS^T Q
//
// Three launches, no atomics, deterministic:
//   bwd_prep   D = rowsum(dO * O) and LSE * log2(e) per query row, padded to
//              whole 128-row blocks (+inf LSE on padded or empty rows, so
//              their P is 0 without a mask).
//   bwd kernel KIND = kBwdDkDv: one task per (b, K/V head, 128-key block):
//              K and V resident, the Q / dO blocks of every query head that
//              reads this K/V head streamed through a ring; S^T = K Q^T and
//              dP^T = V dO^T on tcgen05, P^T and dS^T on the CUDA cores back
//              into TMEM, dV += P^T dO and dK += dS^T Q accumulated in TMEM.
//   bwd kernel KIND = kBwdDq: one task per (b, query head, 128-query block):
//              Q and dO resident, K / V blocks streamed; S = Q K^T,
//              dP = dO V^T, dS, dQ += dS K.
// Both directions are the same loop with the roles of the tiles swapped, so
// they share this code.  Computing dQ in its own pass costs two more GEMMs
// per tile pair (S and dP recomputed) but needs neither the fp32 dQ
// reductions across key blocks nor TMEM beyond 512 columns (S, dP, dK, dV).
//
// Head dims: d_qk = d_v in {64, 128}, and (d_qk, d_v) = (192, 128).  R0 / T0
// (K, Q) have d_qk columns, R1 / T1 (V, dO) d_v columns.
//
// CTA: 320 threads, persistent (grid = SM count).  Each 128-row streamed
// block is taken as two 64-row stages (the forward's two-stage overlap: one
// stage's row warps work while the other stage's GEMMs run):
//   warps 0-3, 4-7  row role of stage 0 / 1: thread = row = TMEM lane (a key
//              for dK/dV, a query for dQ); P and dS for the stage's 64
//              columns, then the epilogue (accumulators -> bf16).
//   warp 8     tcgen05.mma issue (one lane) and TMEM alloc / free.
//   warp 9     TMA loads (one lane).
// TMEM: S_0 [0,64), dP_0 [64,128), S_1 [128,192), dP_1 [192,256),
// accumulator 0 [256, 256+d) (dV or dQ), accumulator 1 [384, 384+d) (dK).
// P^T (dK/dV) or dS (dQ) is written as packed bf16 pairs over the first 32
// columns of S_s, dS^T over the first 32 of dP_s.  At (192, 128) the dK/dV
// accumulators take 128 + 192 columns, so S_s and dP_s share 64 columns per
// stage: S_s lands there, the row warps read it (s_read), dP_s is written
// over it, and P^T / dS^T go to its first / last 32 columns; dV at [128, 256),
// dK at [256, 448).  The dQ kernel at (192, 128) keeps the separate S and dP
// columns with dQ at [256, 448) and reads Q and dO from SMEM (no room for the
// TMEM copies).
//
// Hand-offs (all mbarriers, all waits bounded):
//   res_full / res_empty     resident tiles of a task loaded / no longer read
//   t_full[r] / t_empty[r]   ring slot r of streamed tiles (+ the LSE and D
//                            vectors of the block for dK/dV)
//   s_full[s]                S_s and dP_s of the current block in TMEM (shared
//                            columns: S_s only)
//   s_read[s] (count 128)    shared columns: S_s read by the row warps
//   dp_full[s]               shared columns: dP_s in TMEM
//   p_ready[s] (count 128)   P / dS of stage s written to TMEM
//   acc_done                 the task's accumulators are final
//   acc_free (count 256)     the epilogue of both stages has read them
#pragma once
#include "fa_kernel.cuh"

namespace fa {

enum : int { kBwdDkDv = 0, kBwdDq = 1 };
constexpr int kBwdThreads = 320;

struct BwdParams {
  CUtensorMap tm_r0, tm_r1;  // resident tiles: (K, V) for dK/dV, (Q, dO) for dQ; 4-D (d, H, S, B)
  CUtensorMap tm_t0, tm_t1;  // streamed tiles: (Q, dO) for dK/dV, (K, V) for dQ
  const float* l2;           // [B, Hq, sq_pad]: LSE * log2(e), +inf on padded / empty rows (varlen:
                             // [Hq, vec_hstride], each sequence's padded rows at its offset)
  const float* dvec;         // the same layout: D = rowsum(dO * O), 0 on padded rows
  uint16_t* out0;            // dV (dK/dV) or dQ, bf16 bits
  uint16_t* out1;            // dK (dK/dV)
  unsigned int* status;
  int B, Hq, Hkv, Sq, Sk, sq_pad, ratio;
  int causal;
  int mq, nk;                // ceil(Sq / 128), ceil(Sk / 128)
  int units, blocks;         // tasks = units * blocks: (b, head) units x 128-row blocks
  int section_units;         // causal order: units per L2 section
  // paired causal order (0 = the plain order): blocks of pair_grid heavy tasks
  // followed by their complements (heaviness ranks q and blocks - 1 - q of a
  // unit), then the pair_r pairs left over, heavy tasks first
  int pair_grid, pair_body, pair_r;
  float scale, scale_log2;
  unsigned long long timeout_ns;
  int debug_flags;           // kDebugSkipPArrive: the row warps never signal p_ready (failure-path test)
  uint64_t* trace;           // VAR & kVarTrace: [trace_ctas][kTraceTracks][1 + trace_cap] words
  int trace_ctas;            // CTAs 0 .. trace_ctas-1 record
  int trace_cap;             // records kept per track
  int vec_hstride;           // l2 / dvec elements between query heads (fixed-length: sq_pad)
  // variable-length batches (VAR & kBwdVarlen): this kernel's task records,
  // written on the device by the planning kernel, and their count
  const VarlenTask* vtasks;
  const int* vcount;
};

// VAR bit of the variable-length build (the event log is bit kVarTrace)
constexpr int kBwdVarlen = 8;

// Streamed tiles travel as half-tiles: rows 64s .. 64s+63 of a 128-row block
// are what stage s reads, so each ring slot holds one stage's half of both
// streamed tensors and is released as soon as that stage's GEMMs are done.
// (With whole-block slots the ring only held two blocks at d = 128 and the
// loader could not fetch far enough ahead to hide the L2 latency.)
template <int DQ, int DV>
struct BwdLayout {
  static_assert((DQ == DV && (DQ == 64 || DQ == 128)) || (DQ == 192 && DV == 128), "backward head dims");
  static constexpr int NCQ = DQ / 64, NCV = DV / 64;
  static constexpr int kTile0 = NCQ * kChunkBytes;  // resident R0 (K or Q): 128 rows x d_qk
  static constexpr int kTile1 = NCV * kChunkBytes;  // resident R1 (V or dO): 128 rows x d_v
  static constexpr int kHalfChunk = 64 * 128;       // 64 rows x 128 B
  static constexpr int kHalf0 = NCQ * kHalfChunk;   // streamed T0 half-tile (Q or K)
  static constexpr int kHalf1 = NCV * kHalfChunk;   // streamed T1 half-tile (dO or V)
  static constexpr int kVecH = 64 * 4;              // 64 fp32
  static constexpr int kSlot = kHalf0 + kHalf1;     // T0 half, T1 half (1024-aligned)
  static constexpr int kMaxSmem = 232448;
  static constexpr int NSLOT_fit = (kMaxSmem - kTile0 - kTile1 - 2048 - 1024) / (kSlot + 2 * kVecH);
  static constexpr int NSLOT = NSLOT_fit > 8 ? 8 : NSLOT_fit;
  // three half-slots keep one block ahead of the GEMMs (the next half of a
  // stage loads into the slot its own previous accumulating GEMMs release)
  static_assert(NSLOT >= 3, "ring depth");
  static constexpr int oR0 = 0;
  static constexpr int oR1 = kTile0;
  static constexpr int oRing = kTile0 + kTile1;             // slot r: T0 half, T1 half
  static constexpr int oVec = oRing + NSLOT * kSlot;        // slot r: L2 vector (64), D vector (64)
  static constexpr int oBar = oVec + NSLOT * 2 * kVecH;
  static constexpr int bResFull = 0;
  static constexpr int bResEmpty = 1;
  static constexpr int bTFull = 2;               // [NSLOT]
  static constexpr int bTEmpty = 2 + NSLOT;      // [NSLOT]
  static constexpr int bSFull = 2 + 2 * NSLOT;   // [2] per stage
  static constexpr int bPReady = bSFull + 2;      // [2] per stage, count 128
  static constexpr int bAccDone = bSFull + 4;
  static constexpr int bAccFree = bSFull + 5;     // count 256
  static constexpr int bDrain = bSFull + 6;
  static constexpr int bAReady = bSFull + 7;     // dQ: Q and dO copied into TMEM (count 256)
  static constexpr int bSRead = bSFull + 8;      // [2] shared S / dP columns: S read (count 128)
  static constexpr int bDpFull = bSFull + 10;    // [2] shared S / dP columns: dP in TMEM
  static constexpr int kNumBars = bDpFull + 2;
  static constexpr int oMisc = oBar + kNumBars * 8;  // [0] TMEM base, [1] abort flag
  static constexpr int kBytes = oMisc + 16;
  static constexpr int kDynSmem = kBytes + 1024;
  static_assert(kDynSmem <= kMaxSmem, "shared memory budget");
  static __device__ __forceinline__ uint32_t slot_off(int r) { return oRing + r * kSlot; }
  static __device__ __forceinline__ uint32_t vec_off(int r) { return oVec + r * 2 * kVecH; }
};

// TMEM column plan of a kernel: S_s and dP_s share 64 columns (dK/dV with
// d_qk + d_v > 256), or S_s at 128 s and dP_s at 128 s + 64; the accumulators
// (dV then dK, or dQ); the dQ kernel's TMEM copies of Q and dO (when they fit).
template <int DQ, int DV, int KIND>
struct BwdCols {
  static constexpr bool kShare = KIND == kBwdDkDv && DQ + DV > 256;
  static constexpr bool kTmemA = KIND == kBwdDq && DQ + DV <= 256;
  static constexpr uint32_t kAcc0 = kShare ? 128u : 256u;  // dV (dK/dV) or dQ
  static constexpr uint32_t kAcc1 = kShare ? 256u : 384u;  // dK
  static constexpr uint32_t kQCol = 384u, kOCol = 448u;    // dQ kernel, kTmemA only
  static_assert(KIND != kBwdDkDv || kAcc1 + DQ <= 512, "dK accumulator");
  static_assert(KIND != kBwdDq || kAcc0 + DQ <= (kTmemA ? kQCol : 512u), "dQ accumulator");
  static __device__ __forceinline__ uint32_t s_col(int s) { return static_cast<uint32_t>((kShare ? 64 : 128) * s); }
  static __device__ __forceinline__ uint32_t p_col(int s) {
    return kShare ? static_cast<uint32_t>(64 * s) : static_cast<uint32_t>(128 * s + 64);
  }
  // where P^T (dK/dV) or dS (dQ) and dS^T (dK/dV) are written: the first 32
  // columns of S_s / dP_s, or the two halves of the shared columns
  static __device__ __forceinline__ uint32_t pt_col(int s) { return s_col(s); }
  static __device__ __forceinline__ uint32_t dst_col(int s) { return kShare ? s_col(s) + 32u : p_col(s); }
};

enum : unsigned int {
  kSiteBwdRowS = 601,
  kSiteBwdRowAcc = 602,
  kSiteBwdRowDp = 603,
  kSiteBwdMmaRes = 611,
  kSiteBwdMmaT = 612,
  kSiteBwdMmaP = 613,
  kSiteBwdMmaAcc = 614,
  kSiteBwdMmaDrain = 615,
  kSiteBwdMmaSRead = 616,
  kSiteBwdLoadRes = 621,
  kSiteBwdLoadT = 622,
  kSiteBwdLoadDrain = 623,
};

// One task of either direction.
struct BwdTask {
  int b, h;      // batch (sequence); K/V head (dK/dV) or query head (dQ)
  int blk;       // 128-row block of the resident tiles
  int it0;       // dK/dV: first query block; dQ: 0
  int nit;       // streamed blocks (dK/dV: ratio query heads x (mq - it0) blocks)
  // variable-length batches only (the fixed-length kernels read the
  // problem's values from the parameters instead: BwdSeq)
  int sq, sk;    // the sequence's query and key counts
  int res_r0, str_r0;  // first row of the sequence in the resident / streamed TMA views
  int qbase, kbase;    // row of the sequence's first query / key in q, dq / k, dk, dv
  int vbase;           // l2 / dvec index of the sequence's row 0 of query head 0
};

// The sequence a task belongs to: the task record's values (VARLEN) or the
// fixed-length problem's.
template <bool VARLEN>
struct BwdSeq {
  const BwdParams& p;
  const BwdTask& k;
  __device__ __forceinline__ int sq() const { return VARLEN ? k.sq : p.Sq; }
  __device__ __forceinline__ int sk() const { return VARLEN ? k.sk : p.Sk; }
  __device__ __forceinline__ int mq() const { return VARLEN ? (k.sq + kBM - 1) / kBM : p.mq; }
  __device__ __forceinline__ int nk() const { return VARLEN ? (k.sk + kBN - 1) / kBN : p.nk; }
  __device__ __forceinline__ int bc() const { return VARLEN ? 0 : k.b; }                  // TMA batch coordinate
  __device__ __forceinline__ int res_r0() const { return VARLEN ? k.res_r0 : 0; }      // TMA row offsets
  __device__ __forceinline__ int str_r0() const { return VARLEN ? k.str_r0 : 0; }
  __device__ __forceinline__ int64_t qbase() const { return VARLEN ? k.qbase : static_cast<int64_t>(k.b) * p.Sq; }
  __device__ __forceinline__ int64_t kbase() const { return VARLEN ? k.kbase : static_cast<int64_t>(k.b) * p.Sk; }
  __device__ __forceinline__ int64_t vbase() const {
    return VARLEN ? k.vbase : static_cast<int64_t>(k.b) * p.Hq * p.vec_hstride;
  }
};

// Fixed-length task t: its batch, head and block, and the problem-wide
// fields.  Units are (b, head) pairs; tasks of a unit cover its 128-row
// blocks.  Non-causal: unit by unit.  Causal: sections of `section_units`
// units whose streamed tiles fit in L2 together, heaviest block first inside
// a section (for dK/dV the first key blocks, which every later query sees;
// for dQ the last query blocks, which see every earlier key).  With the
// paired order (an even block count, static assignment over pair_grid CTAs)
// the task of heaviness rank q and its complement blocks - 1 - q, whose
// streamed blocks sum to a constant, run on one CTA in consecutive waves.
template <int KIND>
__device__ __forceinline__ void bwd_task_fixed(const BwdParams& p, int t, BwdTask& k) {
  const int M = p.blocks;
  int unit, q;
  if (!p.causal) {
    unit = t / M;
    q = t - unit * M;
  } else if (p.pair_grid > 0) {
    const int G = p.pair_grid;
    bool light;
    if (t < p.pair_body) {
      const int blk = t / (2 * G);
      const int w = t - blk * 2 * G;
      light = w >= G;
      t = blk * G + (light ? w - G : w);
    } else {
      const int tt = t - p.pair_body;
      light = tt >= p.pair_r;
      t = p.pair_body / 2 + (light ? tt - p.pair_r : tt);
    }
    // pair t: the heavier half (ranks 0 .. M/2 - 1) in section order
    const int Mh = M / 2;
    const int su = p.section_units;
    const int section = t / (su * Mh);
    const int first = section * su;
    int in_section = p.units - first;
    if (in_section > su) in_section = su;
    const int idx = t - section * su * Mh;
    q = idx / in_section;
    unit = first + (idx - q * in_section);
    if (light) q = M - 1 - q;
  } else {
    const int su = p.section_units;
    const int section = t / (su * M);
    const int first = section * su;
    int in_section = p.units - first;
    if (in_section > su) in_section = su;
    const int idx = t - section * su * M;
    q = idx / in_section;  // heaviness rank inside the section
    unit = first + (idx - q * in_section);
  }
  const int H = KIND == kBwdDkDv ? p.Hkv : p.Hq;
  k.b = unit / H;
  k.h = unit - k.b * H;
  // key block, heaviest (lowest) first; or query block, heaviest (highest) first under the mask
  k.blk = KIND == kBwdDkDv ? q : (p.causal ? M - 1 - q : q);
}

// Task t, and the streamed blocks it visits.  Variable-length batches: the
// planning kernel's record t (sequences longest first).  Fixed length: see
// bwd_task_fixed.
template <int KIND, bool VARLEN>
__device__ __forceinline__ BwdTask bwd_task(const BwdParams& p, int t) {
  BwdTask k;
  if constexpr (VARLEN) {
    // record: sequence, head, block, padded row offset; q_row0, sq, k_row0, sk
    const int4* r = reinterpret_cast<const int4*>(p.vtasks + t);
    const int4 a = r[0], c = r[1];
    k.b = a.x, k.h = a.y, k.blk = a.z;
    k.vbase = a.w;
    k.qbase = c.x, k.sq = c.y, k.kbase = c.z, k.sk = c.w;
    k.res_r0 = KIND == kBwdDkDv ? c.z : c.x;
    k.str_r0 = KIND == kBwdDkDv ? c.x : c.z;
  } else {
    bwd_task_fixed<KIND>(p, t, k);
  }
  const BwdSeq<VARLEN> sq{p, k};
  if (KIND == kBwdDkDv) {
    int first_q = 0;
    if (p.causal) {  // the first query that sees key blk * 128: q >= k - (Sk - Sq)
      const int qmin = k.blk * kBN - (sq.sk() - sq.sq());
      first_q = qmin > 0 ? qmin / kBM : 0;
    }
    k.it0 = first_q;
    k.nit = first_q < sq.mq() ? p.ratio * (sq.mq() - first_q) : 0;
  } else {
    k.it0 = 0;
    int n = sq.nk();
    if (p.causal) {
      int last = (k.blk + 1) * kBM;
      if (last > sq.sq()) last = sq.sq();
      const int64_t max_key = static_cast<int64_t>(last - 1) + sq.sk() - sq.sq();
      n = max_key < 0 ? 0 : static_cast<int>(max_key / kBN + 1);
      if (n > sq.nk()) n = sq.nk();
    }
    k.nit = k.blk * kBM < sq.sq() ? n : 0;
  }
  return k;
}


// Tasks of this kernel: the fixed-length grid of units x blocks, or the
// planning kernel's count.
template <bool VARLEN>
__device__ __forceinline__ int bwd_task_count(const BwdParams& p) {
  if constexpr (VARLEN) return *p.vcount;
  else return p.units * p.blocks;
}

// Streamed block `it` of a task: for dK/dV the query head and query block,
// for dQ the key block.
struct BwdIter {
  int head;  // head of the streamed tiles' view
  int blk;   // their 128-row block
};

template <int KIND, bool VARLEN>
__device__ __forceinline__ BwdIter bwd_iter(const BwdParams& p, const BwdTask& k, int it) {
  BwdIter r;
  if (KIND == kBwdDkDv) {
    const int nq = BwdSeq<VARLEN>{p, k}.mq() - k.it0;
    const int hh = it / nq;
    r.head = k.h * p.ratio + hh;
    r.blk = k.it0 + (it - hh * nq);
  } else {
    r.head = k.h / p.ratio;  // the K/V head the query head reads
    r.blk = it;
  }
  return r;
}

// ---------------------------------------------------------------------------
// S-like GEMM over half a streamed tile: D[128 x 64] = A[128 x D] B[64 x D]^T,
// A and B K-major in SMEM (B = rows 64s .. 64s+63 of the streamed tile: the
// 128-byte swizzle repeats every 8 rows, so the offset keeps its phase).
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void issue_qk64(uint32_t d_tmem, uint32_t a_addr, uint32_t b_addr, uint32_t leader) {
  constexpr uint32_t kIdesc = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {  // A: whole tile, 64-column chunks 16 KB apart; B: half-tile, 8 KB apart
    const uint32_t ao = opaque_u32(static_cast<uint32_t>(c * kChunkBytes));
    const uint32_t bo = opaque_u32(static_cast<uint32_t>(c * 64 * 128));
    mma_ss_x4<2, 2>(d_tmem, smem_desc_sw128(a_addr + ao, 16, 1024), smem_desc_sw128(b_addr + bo, 16, 1024), kIdesc,
                    c != 0 ? 1u : 0u, leader);
  }
}

// The same with A in TMEM (the dQ kernel's Q or dO, D / 2 columns of packed
// bf16 pairs): only B is read from SMEM.
template <int D>
__device__ __forceinline__ void issue_ts_qk64(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_addr, uint32_t leader) {
  constexpr uint32_t kIdesc = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    const uint32_t bo = opaque_u32(static_cast<uint32_t>(c * 64 * 128));
    mma_ts_x4<2>(d_tmem, a_tmem + static_cast<uint32_t>(32 * c), smem_desc_sw128(b_addr + bo, 16, 1024), kIdesc,
                 c != 0 ? 1u : 0u, leader);
  }
}

// Accumulating GEMM over one stage: D[128 x D] (+)= A[128 x 64] B[64 x D],
// A in TMEM (32 columns of packed bf16 pairs), B a streamed half-tile read
// MN-major (16 rows per step; its 64-column chunks 8 KB apart).
template <int D>
__device__ __forceinline__ void issue_pv64(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_addr, bool accumulate,
                                           uint32_t leader) {
  constexpr uint32_t kIdesc = idesc_bf16_f32(128, D, false, true);
  constexpr uint32_t kStep = 16 * 128 >> 4;  // 16 rows, in 16-byte units
  mma_ts_x4<kStep>(d_tmem, a_tmem, smem_desc_sw128(opaque_u32(b_addr), 64 * 128, 1024), kIdesc,
                   accumulate ? 1u : 0u, leader);
}

// ---------------------------------------------------------------------------
// row role (warpgroup s = stage s): thread = row = TMEM lane
// ---------------------------------------------------------------------------
// Per streamed block, stage s takes its 64 columns (rows 64s .. 64s+63 of the
// streamed tile): P = 2^(S * scale * log2(e) - LSE * log2(e)) on the visible
// entries (0 elsewhere), dS = P (dP - D).  dK/dV: rows are keys, columns
// queries (LSE and D per column, from the block's vectors in the ring slot);
// dQ: rows are queries (LSE and D per row), columns keys.
template <int DQ, int DV, int KIND, bool CAUSAL, int VAR>
__device__ __forceinline__ void bwd_row_role(const BwdParams& p, const int stage, const uint32_t tmem,
                                             const uint32_t sbase, const uint8_t* smem, const WaitCtx& wc) {
  constexpr bool VARLEN = (VAR & kBwdVarlen) != 0;
  using L = BwdLayout<DQ, DV>;
  using C = BwdCols<DQ, DV, KIND>;
  const int t = threadIdx.x - 128 * stage;
  const uint32_t lane_off = static_cast<uint32_t>(t & ~31) << 16;
  const uint32_t tS = tmem + lane_off + C::s_col(stage);  // S_s, then P^T (dK/dV) or dS (dQ) over its first 32 columns
  const uint32_t tP = tmem + lane_off + C::p_col(stage);  // dP_s, then dS^T (dK/dV) over its first 32 columns
  const uint32_t bar0 = sbase + L::oBar;
  uint32_t dp_phase = 0;  // shared S / dP columns
  const float sl2 = p.scale_log2;
  const int cb = 64 * stage;  // first column of this stage inside the streamed block
  uint32_t s_phase = 0, acc_phase = 0;
  int slot_it = 0;
  const int num_tasks = bwd_task_count<VARLEN>(p);

  uint32_t res_phase = 0;
  Tracer<(VAR & kVarTrace) != 0, -1> tr;  // track = stage
  tr.init(p, t == 0, stage);
  for (int task = blockIdx.x; task < num_tasks; task += gridDim.x) {
    const BwdTask tk = bwd_task<KIND, VARLEN>(p, task);
    const BwdSeq<VARLEN> sq{p, tk};
    const int row = tk.blk * kBM + t;  // key (dK/dV) or query (dQ)
    tr.ev(p, kEvBrTask, static_cast<uint32_t>(task));
    if constexpr (C::kTmemA) {
      // stage s copies its resident tile (Q or dO, row t, 128-byte swizzled
      // in SMEM) into TMEM as packed bf16 pairs.  The previous task's
      // epilogue waited for all its MMAs, so these columns are free.
      if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8u * L::bResFull, res_phase, wc, kSiteBwdRowS))) return;
      res_phase ^= 1u;
      const uint8_t* tile = smem + (stage == 0 ? L::oR0 : L::oR1);
      const uint32_t tA = tmem + lane_off + (stage == 0 ? C::kQCol : C::kOCol);
#pragma unroll
      for (int c = 0; c < L::NCQ; ++c) {
        const uint4* src = reinterpret_cast<const uint4*>(tile + c * kChunkBytes + t * 128);
        uint32_t w[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 v = src[q ^ (t & 7)];
          w[4 * q] = v.x, w[4 * q + 1] = v.y, w[4 * q + 2] = v.z, w[4 * q + 3] = v.w;
        }
        tmem_st32(tA + static_cast<uint32_t>(32 * c), w);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar0 + 8u * L::bAReady);
    }
    float l2_row = 0.f, d_row = 0.f;
    if (KIND == kBwdDq) {  // row < sq_pad: the block lies inside the padded rows
      const int64_t vi = sq.vbase() + static_cast<int64_t>(tk.h) * p.vec_hstride + row;
      l2_row = p.l2[vi];
      d_row = p.dvec[vi];
    }
    for (int it = 0; it < tk.nit; ++it, ++slot_it) {
      const BwdIter bi = bwd_iter<KIND, VARLEN>(p, tk, it);
      const int slot = (2 * slot_it + stage) % L::NSLOT;  // this stage's half of block it
      tr.ev(p, kEvBrWait, static_cast<uint32_t>(it));
      if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8u * (L::bSFull + stage), s_phase, wc, kSiteBwdRowS))) {
        tr.finish(p);
        return;
      }
      s_phase ^= 1u;
      tc_fence_after();
      tr.ev(p, kEvBrS, static_cast<uint32_t>(it));

      // visible columns c (0 .. 63 of this stage) in [cmin, cmax]
      int cmin = 0, cmax = 63;
      bool row_ok = true;
      if (KIND == kBwdDkDv) {
        row_ok = row < sq.sk();
        if (CAUSAL) cmin = row - (sq.sk() - sq.sq()) - bi.blk * kBM - cb;  // query q sees key k iff q >= k - (Sk - Sq)
      } else {
        cmax = min(63, sq.sk() - 1 - bi.blk * kBN - cb);  // keys < Sk
        if (CAUSAL) cmax = min(cmax, row + (sq.sk() - sq.sq()) - bi.blk * kBN - cb);
      }
      // the block's LSE and D per column (dK/dV), read four at a time (every
      // lane reads the same 16 bytes: one shared-memory wavefront per four
      // columns, which the tensor cores' operand reads share)
      const float4* l2v = reinterpret_cast<const float4*>(smem + L::vec_off(slot));
      const float4* dvv = l2v + 16;

      uint32_t r[64];
      tmem_ld64_wait(tS, r);
      float pr[64];
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 l4 = KIND == kBwdDkDv ? l2v[c4] : make_float4(l2_row, l2_row, l2_row, l2_row);
        const float lse2[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = 4 * c4 + j;
          const bool vis = row_ok && c >= cmin && c <= cmax;
          pr[c] = vis ? ex2_approx(__uint_as_float(r[c]) * sl2 - lse2[j]) : 0.f;
        }
      }
      if constexpr (C::kShare) {
        // S is in registers: dP_s may now be written over it
        tc_fence_before();
        mbar_arrive(bar0 + 8u * (L::bSRead + stage));
        if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8u * (L::bDpFull + stage), dp_phase, wc, kSiteBwdRowDp)))
          return;
        dp_phase ^= 1u;
        tc_fence_after();
        // dS^T = P^T (dP^T - D) from the whole of dP_s (loaded before either
        // half of the columns is overwritten), then P^T and dS^T over them
        uint32_t dp[64];
        tmem_ld64_wait(tP, dp);
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // 16 packed columns of each at a time
          uint32_t pk[16], dk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c0 = 32 * h + 2 * i;
            const float4 d4 = dvv[c0 / 4];
            const float d0 = (i & 1) ? d4.z : d4.x, d1 = (i & 1) ? d4.w : d4.y;
            pk[i] = pack_bf16x2(pr[c0], pr[c0 + 1]);
            dk[i] = pack_bf16x2(pr[c0] * (__uint_as_float(dp[c0]) - d0), pr[c0 + 1] * (__uint_as_float(dp[c0 + 1]) - d1));
          }
          tmem_st16(tmem + lane_off + C::pt_col(stage) + static_cast<uint32_t>(16 * h), pk);
          tmem_st16(tmem + lane_off + C::dst_col(stage) + static_cast<uint32_t>(16 * h), dk);
        }
      } else {
        if (KIND == kBwdDkDv) {  // P^T for dV += P^T dO
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) pk[i] = pack_bf16x2(pr[2 * i], pr[2 * i + 1]);
          tmem_st32(tS, pk);
        }
        // dS = P (dP - D), 32 columns at a time, onto columns 16q .. 16q+15 of
        // dP (dK/dV) or S (dQ), all of them read already
        const uint32_t tDst = KIND == kBwdDkDv ? tP : tS;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t dp[32];
          tmem_ld32_wait(tP + static_cast<uint32_t>(32 * q), dp);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c0 = 32 * q + 2 * i;
            float d0 = d_row, d1 = d_row;
            if (KIND == kBwdDkDv) {
              const float4 d4 = dvv[c0 / 4];
              d0 = (i & 1) ? d4.z : d4.x;
              d1 = (i & 1) ? d4.w : d4.y;
            }
            pk[i] = pack_bf16x2(pr[c0] * (__uint_as_float(dp[2 * i]) - d0),
                                pr[c0 + 1] * (__uint_as_float(dp[2 * i + 1]) - d1));
          }
          tmem_st16(tDst + static_cast<uint32_t>(16 * q), pk);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      if (!(p.debug_flags & kDebugSkipPArrive)) mbar_arrive(bar0 + 8u * (L::bPReady + stage));
      tr.ev(p, kEvBrP, static_cast<uint32_t>(it));
    }

    // epilogue: dK/dV: stage 0 writes dV, stage 1 dK (scaled); dQ: stage s
    // writes columns [s D/2, (s+1) D/2) (scaled)
    if (tk.nit > 0) {
      if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8u * L::bAccDone, acc_phase, wc, kSiteBwdRowAcc))) {
        tr.finish(p);
        return;
      }
      acc_phase ^= 1u;
      tc_fence_after();
    }
    tr.ev(p, kEvBrAcc, static_cast<uint32_t>(task));
    const bool store = KIND == kBwdDkDv ? row < sq.sk() : row < sq.sq();
    uint16_t* dst;
    float mult;
    uint32_t tA;
    int c_lo, c_hi;
    if (KIND == kBwdDkDv) {
      const int64_t rr = (sq.kbase() + row) * p.Hkv + tk.h;
      dst = stage == 0 ? p.out0 + rr * DV : p.out1 + rr * DQ;  // dV, dK
      mult = stage == 0 ? 1.f : p.scale;
      tA = tmem + lane_off + (stage == 0 ? C::kAcc0 : C::kAcc1);
      c_lo = 0, c_hi = stage == 0 ? DV : DQ;
    } else {
      dst = p.out0 + ((sq.qbase() + row) * p.Hq + tk.h) * DQ;
      mult = p.scale;
      tA = tmem + lane_off + C::kAcc0;
      c_lo = stage * (DQ / 2), c_hi = c_lo + DQ / 2;
    }
#pragma unroll 1
    for (int c = c_lo; c < c_hi; c += 32) {
      uint32_t v[32];
      if (tk.nit > 0) {  // uniform across the CTA: the loads stay warp-collective
        tmem_ld32_wait(tA + static_cast<uint32_t>(c), v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0u;
      }
      if (store) {
        uint4* o4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]) * mult, __uint_as_float(v[8 * q + 1]) * mult);
          w.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]) * mult, __uint_as_float(v[8 * q + 3]) * mult);
          w.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]) * mult, __uint_as_float(v[8 * q + 5]) * mult);
          w.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]) * mult, __uint_as_float(v[8 * q + 7]) * mult);
          o4[q] = w;
        }
      }
    }
    tc_fence_before();
    mbar_arrive(bar0 + 8u * L::bAccFree);
    tr.ev(p, kEvBrEpi, static_cast<uint32_t>(task));
  }
  tr.finish(p);
}

// ---------------------------------------------------------------------------
// MMA issue (warp 8; lane 0 issues)
// ---------------------------------------------------------------------------
// Per streamed block j and stage s: the accumulating GEMMs of (j, s) as soon
// as stage s has written P / dS, then S and dP of (j+1, s), so one stage's
// row warps work while the other stage's GEMMs run.
template <int DQ, int DV, int KIND, int VAR>
__device__ __forceinline__ void bwd_mma_role(const BwdParams& p, const uint32_t tmem, const uint32_t sbase,
                                             const WaitCtx& wc) {
  constexpr bool VARLEN = (VAR & kBwdVarlen) != 0;
  using L = BwdLayout<DQ, DV>;
  using C = BwdCols<DQ, DV, KIND>;
  const uint32_t bar0 = sbase + L::oBar;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  const uint32_t leader = (threadIdx.x & 31) == 0 ? 1u : 0u;
  auto wait = [&](uint32_t b, uint32_t parity, unsigned site) {
    return __all_sync(0xffffffffu, mbar_wait(b, parity, wc, site));
  };
  uint32_t res_phase = 0, free_phase = 0, a_phase = 0, p_phase[2] = {0u, 0u}, sr_phase[2] = {0u, 0u};
  int slot_it = 0;  // streamed blocks consumed; block i's stage-s half sits in slot (2 i + s) % NSLOT
  const int num_tasks = bwd_task_count<VARLEN>(p);
  const uint32_t r0 = sbase + L::oR0, r1 = sbase + L::oR1;
  auto half_slot = [&](int blk_it, int s) { return (2 * blk_it + s) % L::NSLOT; };
  auto half_parity = [&](int blk_it, int s) { return static_cast<uint32_t>((2 * blk_it + s) / L::NSLOT) & 1u; };
  // S_s and dP_s of the half in `slot`; with shared columns only S_s here
  // (dP_s follows once the row warps have read S_s: issue_dp)
  auto issue_sdp = [&](int s, int slot) {
    const uint32_t t0 = sbase + L::slot_off(slot), t1 = t0 + L::kHalf0;
    if constexpr (C::kTmemA) {
      issue_ts_qk64<DQ>(tmem + C::s_col(s), tmem + C::kQCol, t0, leader);  // S_s  = Q K_s^T
      issue_ts_qk64<DV>(tmem + C::p_col(s), tmem + C::kOCol, t1, leader);  // dP_s = dO V_s^T
    } else {
      issue_qk64<DQ>(tmem + C::s_col(s), r0, t0, leader);                    // S_s  = R0 T0_s^T
      if constexpr (!C::kShare) issue_qk64<DV>(tmem + C::p_col(s), r1, t1, leader);  // dP_s = R1 T1_s^T
    }
    mma_commit(bar(L::bSFull + s), leader);
  };
  // shared columns: dP_s over S_s once the row warps have read it
  auto issue_dp = [&](int s, int slot) -> bool {
    if (!wait(bar(L::bSRead + s), sr_phase[s], kSiteBwdMmaSRead)) return false;
    sr_phase[s] ^= 1u;
    tc_fence_after();
    issue_qk64<DV>(tmem + C::p_col(s), r1, sbase + L::slot_off(slot) + L::kHalf0, leader);  // dP_s = R1 T1_s^T
    mma_commit(bar(L::bDpFull + s), leader);
    return true;
  };

  Tracer<(VAR & kVarTrace) != 0, 3> tr;
  tr.init(p, leader != 0);
  for (int task = blockIdx.x, n = 0; task < num_tasks; task += gridDim.x, ++n) {
    const BwdTask tk = bwd_task<KIND, VARLEN>(p, task);
    if (!wait(bar(L::bResFull), res_phase, kSiteBwdMmaRes)) goto out;
    res_phase ^= 1u;
    tr.ev(p, kEvBmTask, static_cast<uint32_t>(task));
    if (n > 0) {  // the previous task's epilogue has read the accumulators
      if (!wait(bar(L::bAccFree), free_phase, kSiteBwdMmaAcc)) goto out;
      free_phase ^= 1u;
    }
    if constexpr (C::kTmemA) {  // Q and dO of this task are in TMEM
      if (!wait(bar(L::bAReady), a_phase, kSiteBwdMmaRes)) goto out;
      a_phase ^= 1u;
    }
    tc_fence_after();
    if (tk.nit > 0) {
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        if (!wait(bar(L::bTFull + half_slot(slot_it, s)), half_parity(slot_it, s), kSiteBwdMmaT)) goto out;
        tc_fence_after();
        tr.ev(p, kEvBmT, static_cast<uint32_t>(s << 16));
        issue_sdp(s, half_slot(slot_it, s));
        tr.ev(p, kEvBmSdp, static_cast<uint32_t>(s << 16));
      }
      if constexpr (C::kShare) {
#pragma unroll
        for (int s = 0; s < 2; ++s)
          if (!issue_dp(s, half_slot(slot_it, s))) goto out;
      }
    }
    for (int it = 0; it < tk.nit; ++it, ++slot_it) {
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const int slot = half_slot(slot_it, s);
        const uint32_t t0 = sbase + L::slot_off(slot), t1 = t0 + L::kHalf0;
        if (!wait(bar(L::bPReady + s), p_phase[s], kSiteBwdMmaP)) goto out;
        p_phase[s] ^= 1u;
        tc_fence_after();
        tr.ev(p, kEvBmP, static_cast<uint32_t>(s << 16 | it));
        const bool acc = it > 0 || s > 0;
        if (KIND == kBwdDkDv) {
          issue_pv64<DV>(tmem + C::kAcc0, tmem + C::pt_col(s), t1, acc, leader);   // dV += P^T_s dO_s
          issue_pv64<DQ>(tmem + C::kAcc1, tmem + C::dst_col(s), t0, acc, leader);  // dK += dS^T_s Q_s
        } else {
          issue_pv64<DQ>(tmem + C::kAcc0, tmem + C::s_col(s), t0, acc, leader);    // dQ += dS_s K_s
        }
        mma_commit(bar(L::bTEmpty + slot), leader);  // this half is no longer read
        tr.ev(p, kEvBmAcc, static_cast<uint32_t>(s << 16 | it));
        if (it + 1 < tk.nit) {
          const int nslot = half_slot(slot_it + 1, s);
          if (!wait(bar(L::bTFull + nslot), half_parity(slot_it + 1, s), kSiteBwdMmaT)) goto out;
          tc_fence_after();
          tr.ev(p, kEvBmT, static_cast<uint32_t>(s << 16 | (it + 1)));
          issue_sdp(s, nslot);
          tr.ev(p, kEvBmSdp, static_cast<uint32_t>(s << 16 | (it + 1)));
        }
      }
      if constexpr (C::kShare) {  // dP of the next block, once each stage has read its S
        if (it + 1 < tk.nit) {
#pragma unroll
          for (int s = 0; s < 2; ++s)
            if (!issue_dp(s, half_slot(slot_it + 1, s))) goto out;
        }
      }
    }
    if (tk.nit > 0) mma_commit(bar(L::bAccDone), leader);
    mma_commit(bar(L::bResEmpty), leader);
  }
out:
  mma_commit(bar(L::bDrain), leader);
  mbar_drain_wait(bar(L::bDrain), 0u, wc, kSiteBwdMmaDrain);
  tr.finish(p);
}

// ---------------------------------------------------------------------------
// TMA loads (warp 9, one lane)
// ---------------------------------------------------------------------------
template <int DQ, int DV, int KIND, int VAR>
__device__ __forceinline__ void bwd_load_role(const BwdParams& p, const uint32_t sbase, const WaitCtx& wc) {
  constexpr bool VARLEN = (VAR & kBwdVarlen) != 0;
  using L = BwdLayout<DQ, DV>;
  const uint32_t bar0 = sbase + L::oBar;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t res_uses = 0;
  int half_it = 0;  // streamed half-tiles issued
  const int num_tasks = bwd_task_count<VARLEN>(p);
  tma_prefetch_desc(&p.tm_r0);
  tma_prefetch_desc(&p.tm_r1);
  tma_prefetch_desc(&p.tm_t0);
  tma_prefetch_desc(&p.tm_t1);

  Tracer<(VAR & kVarTrace) != 0, 4> tr;
  tr.init(p, true);
  for (int task = blockIdx.x; task < num_tasks; task += gridDim.x) {
    const BwdTask tk = bwd_task<KIND, VARLEN>(p, task);
    const BwdSeq<VARLEN> sq{p, tk};
    tr.ev(p, kEvBlTask, static_cast<uint32_t>(task));
    if (res_uses > 0 && !mbar_wait(bar(L::bResEmpty), (res_uses - 1u) & 1u, wc, kSiteBwdLoadRes)) goto out;
    mbar_arrive_expect_tx(bar(L::bResFull), static_cast<uint32_t>(L::kTile0 + L::kTile1));
    for (int c = 0; c < L::NCQ; ++c)
      tma_load_4d(sbase + L::oR0 + c * kChunkBytes, &p.tm_r0, bar(L::bResFull), c * 64, tk.h,
                  sq.res_r0() + tk.blk * kBM, sq.bc());
    for (int c = 0; c < L::NCV; ++c)
      tma_load_4d(sbase + L::oR1 + c * kChunkBytes, &p.tm_r1, bar(L::bResFull), c * 64, tk.h,
                  sq.res_r0() + tk.blk * kBM, sq.bc());
    ++res_uses;
    for (int it = 0; it < tk.nit; ++it) {
      const BwdIter bi = bwd_iter<KIND, VARLEN>(p, tk, it);
      for (int s = 0; s < 2; ++s, ++half_it) {  // stage s's half: rows 64s .. 64s+63 of the block
        const int slot = half_it % L::NSLOT;
        if (half_it >= L::NSLOT &&
            !mbar_wait(bar(L::bTEmpty + slot), static_cast<uint32_t>(half_it / L::NSLOT - 1) & 1u, wc,
                       kSiteBwdLoadT))
          goto out;
        const uint32_t t0 = sbase + L::slot_off(slot), t1 = t0 + L::kHalf0;
        const uint32_t fb = bar(L::bTFull + slot);
        const int row = bi.blk * kBM + 64 * s;
        mbar_arrive_expect_tx(fb, static_cast<uint32_t>(L::kHalf0 + L::kHalf1) +
                                      (KIND == kBwdDkDv ? 2u * L::kVecH : 0u));
        for (int c = 0; c < L::NCQ; ++c)
          tma_load_4d(t0 + c * L::kHalfChunk, &p.tm_t0, fb, c * 64, bi.head, sq.str_r0() + row, sq.bc());
        for (int c = 0; c < L::NCV; ++c)
          tma_load_4d(t1 + c * L::kHalfChunk, &p.tm_t1, fb, c * 64, bi.head, sq.str_r0() + row, sq.bc());
        if (KIND == kBwdDkDv) {  // LSE and D of these 64 queries (whole padded blocks: always in range)
          const int64_t vi = sq.vbase() + static_cast<int64_t>(bi.head) * p.vec_hstride + row;
          const uint32_t vdst = sbase + L::vec_off(slot);
          bulk_load(vdst, p.l2 + vi, L::kVecH, fb);
          bulk_load(vdst + L::kVecH, p.dvec + vi, L::kVecH, fb);
        }
        tr.ev(p, kEvBlT, static_cast<uint32_t>(half_it));
      }
    }
  }
out:
  if (res_uses > 0) mbar_drain_wait(bar(L::bResFull), (res_uses - 1u) & 1u, wc, kSiteBwdLoadDrain);
  for (int i = 0; i < L::NSLOT && i < half_it; ++i) {
    const uint32_t uses = static_cast<uint32_t>((half_it - i + L::NSLOT - 1) / L::NSLOT);
    mbar_drain_wait(bar(L::bTFull + i), (uses - 1u) & 1u, wc, kSiteBwdLoadDrain);
  }
  tr.finish(p);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// VAR: 0, or kVarTrace for the event-log build
template <int DQ, int DV, int KIND, bool CAUSAL, int VAR = 0>
__global__ void __launch_bounds__(kBwdThreads, 1) fa_bwd_kernel(const __grid_constant__ BwdParams p) {
  using L = BwdLayout<DQ, DV>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::oMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::oMisc + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    const uint32_t b = sbase + L::oBar;
    mbar_init(b + 8 * L::bResFull, 1);
    mbar_init(b + 8 * L::bResEmpty, 1);
    for (int i = 0; i < L::NSLOT; ++i) {
      mbar_init(b + 8 * (L::bTFull + i), 1);
      mbar_init(b + 8 * (L::bTEmpty + i), 1);
    }
    for (int st = 0; st < 2; ++st) {
      mbar_init(b + 8 * (L::bSFull + st), 1);
      mbar_init(b + 8 * (L::bPReady + st), 128);
    }
    mbar_init(b + 8 * L::bAccDone, 1);
    mbar_init(b + 8 * L::bAccFree, 256);
    mbar_init(b + 8 * L::bDrain, 1);
    mbar_init(b + 8 * L::bAReady, 256);
    for (int st = 0; st < 2; ++st) {
      mbar_init(b + 8 * (L::bSRead + st), 128);
      mbar_init(b + 8 * (L::bDpFull + st), 1);
    }
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 8) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  if (warp < 8) {
    bwd_row_role<DQ, DV, KIND, CAUSAL, VAR>(p, warp >> 2, tmem, sbase, smem, wc);
  } else if (warp == 8) {
    bwd_mma_role<DQ, DV, KIND, VAR>(p, tmem, sbase, wc);
    __syncwarp();
  } else if (warp == 9) {
    if (lane == 0) bwd_load_role<DQ, DV, KIND, VAR>(p, sbase, wc);
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// prep: D = rowsum(dO * O) and LSE * log2(e) per (b, query head, row), rows
// padded to whole 128-row blocks; one warp per row
// ---------------------------------------------------------------------------
// D of one row (elements at `off` of o and dout, D_V of them), summed over
// the warp: every lane returns the total
template <int D>
__device__ __forceinline__ float prep_row_dot(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                                              int64_t off, bool valid) {
  constexpr int kPer = D / 32;  // 2 or 4 bf16 per lane
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
  if (valid) {
    off += lane * kPer;
    uint32_t ow[kPer / 2], gw[kPer / 2];
    if constexpr (kPer == 4) {
      const uint2 a = *reinterpret_cast<const uint2*>(o + off);
      const uint2 g = *reinterpret_cast<const uint2*>(dout + off);
      ow[0] = a.x, ow[1] = a.y, gw[0] = g.x, gw[1] = g.y;
    } else {
      ow[0] = *reinterpret_cast<const uint32_t*>(o + off);
      gw[0] = *reinterpret_cast<const uint32_t*>(dout + off);
    }
#pragma unroll
    for (int w = 0; w < kPer / 2; ++w) {
      acc += __uint_as_float(ow[w] << 16) * __uint_as_float(gw[w] << 16);
      acc += __uint_as_float(ow[w] & 0xffff0000u) * __uint_as_float(gw[w] & 0xffff0000u);
    }
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  return acc;
}

// the row's base-2 LSE: +inf for padded rows and rows with no visible key (P = 0)
__device__ __forceinline__ float prep_row_l2(const float* __restrict__ lse, int64_t i, bool valid) {
  float v = INFINITY;
  if (valid) {
    const float l = lse[i];
    if (l != -INFINITY) v = l * 1.4426950408889634f;
  }
  return v;
}

template <int D>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const uint16_t* __restrict__ o,
                                                          const uint16_t* __restrict__ dout,
                                                          const float* __restrict__ lse, float* __restrict__ l2,
                                                          float* __restrict__ dvec, int B, int Hq, int Sq,
                                                          int sq_pad) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = static_cast<int64_t>(B) * Hq * sq_pad;
  const int64_t step = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += step) {
    const int64_t bh = r / sq_pad;
    const int i = static_cast<int>(r - bh * sq_pad);
    const int64_t b = bh / Hq;
    const int h = static_cast<int>(bh - b * Hq);
    const bool valid = i < Sq;
    const float acc = prep_row_dot<D>(o, dout, ((b * Sq + i) * Hq + h) * D, valid);
    if (lane == 0) {
      l2[r] = prep_row_l2(lse, bh * Sq + i, valid);
      dvec[r] = valid ? acc : 0.f;
    }
  }
}

// The same for a variable-length batch, one warp per row of each dQ task
// record (sequence b, query head h, 128-row block; the sequence's padded row
// offset, first row and length): rows at h * vec_hstride + offset + row, LSE
// from [Hq, total_q].
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_prep_varlen_kernel(const uint16_t* __restrict__ o,
                                                                 const uint16_t* __restrict__ dout,
                                                                 const float* __restrict__ lse,
                                                                 float* __restrict__ l2, float* __restrict__ dvec,
                                                                 const VarlenTask* __restrict__ tasks,
                                                                 const int* __restrict__ count, int Hq,
                                                                 int64_t total_q, int vec_hstride) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = static_cast<int64_t>(*count) * kBM;
  const int64_t step = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += step) {
    const int4* rec = reinterpret_cast<const int4*>(tasks + (r / kBM));
    const int4 a = rec[0], c = rec[1];  // b, h, block, offset; q_row0, sq, k_row0, sk
    const int h = a.y;
    const int i = a.z * kBM + static_cast<int>(r % kBM);  // row inside the sequence
    const bool valid = i < c.y;
    const int64_t q = static_cast<int64_t>(c.x) + i;  // row in the packed tensors
    const float acc = prep_row_dot<D>(o, dout, (q * Hq + h) * D, valid);
    if (lane == 0) {
      const int64_t idx = static_cast<int64_t>(h) * vec_hstride + a.w + i;
      l2[idx] = prep_row_l2(lse, h * total_q + q, valid);
      dvec[idx] = valid ? acc : 0.f;
    }
  }
}

}  // namespace fa
