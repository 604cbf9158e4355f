// Exact attention forward for sm_103a: O = softmax(scale * Q K^T) V and the
// per-row log-sum-exp, tiled over K/V blocks with an online softmax so the
// score matrix never reaches HBM.
//
// One persistent CTA per SM, 512 threads in four warpgroups
// ("Flash Attention 4 on Blackwell", sections "The data flow of one K/V
// block" and "Warpgroup roles"):
//   WG0 / WG1 (warps 0-7)  softmax of Q stage 0 / 1: thread = row = TMEM lane;
//                          S is read from TMEM, P (bf16) written back over it.
//   WG2 (warps 8-11)       O correction (rescale O in TMEM when a row's
//                          reference moved) and the epilogue: O / row_sum ->
//                          bf16 -> SMEM -> TMA store, LSE -> global.
//   warp 12                tcgen05.mma issue (one thread) + TMEM alloc/free.
//   warp 13                TMA loads (one thread): Q stages, K/V ring.
// Each task covers two Q tiles (stages) that stream the same K/V blocks, so
// one stage's softmax overlaps the other stage's MMAs.  With VARLEN the
// sequences are packed back to back (rows cu_seqlens[b] ..) and the tasks
// come from a list written by the planning kernel; each task carries its
// sequence's lengths and row offsets.
//
// Modes (one instantiation each): fixed-length; fixed-length with the FMA-pipe
// exp2; varlen (tasks from the planned list, always dynamic); fixed-length
// with dynamic task assignment; split-KV (each task one key range, partial
// O / LSE in fp32 to a workspace, combined afterwards by the merge kernel);
// fixed-length with a direct epilogue (each O row written from registers
// with 32-byte stores instead of SMEM staging and TMA stores, so the
// correction warps return sooner to the next task; the default for
// fixed-length problems, the staged mode on request).
//
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+DV),
// O1 [384,384+DV).  P_s overwrites the first 64 columns of S_s as packed bf16
// pairs.  SMEM: two Q stages, a ring of K/V tiles, a 16 KB O staging tile,
// the softmax -> correction mailbox and the mbarriers.
//
// Hand-offs per stage s and K/V block j (mbarrier names follow the pages'
// "Softmax, correction and barrier hand-off" section):
//   s_full[s]    MMA commit after S_s = Q_s K_j^T            -> softmax
//   corr_full[s] blocks after a task's first: softmax posted
//                acc_scale (right after the row max, before
//                the exponentials)                           -> correction
//   fin_full[s][t & 1]  last block of task t only: row_sum and the
//                reference posted for the epilogue, in one of
//                two slots by task parity                    -> correction
//   p_full[s]    count 256: 128 softmax threads (P written) +
//                128 correction threads (O rescaled or not;
//                for a task's first block: O free, an arrival
//                made as soon as the previous task's epilogue
//                has read O_s out of TMEM)                   -> PV MMA
// The two fin_full slots let the correction warps signal a stage's last block
// without first reading its final statistics (the slot a task writes was read
// two tasks earlier, before the P V that the writer's S depends on); the
// early O-free arrival lets a task's first P V start behind one epilogue, not
// behind both stages' epilogues and the next task's first row maximum.
//   o_done[s]    MMA commit after the stage's last P V of a
//                task                                        -> epilogue
//   task_full[r] / task_empty[r]  (DYN only) the TMA thread takes the next
//                task index from a global counter (atomicAdd) and posts it in
//                ring slot r; every other warp reads it and frees the slot.
// Task assignment: static round-robin (task = blockIdx.x + k * gridDim.x), or
// with DYN dynamic, in list order, to whichever CTA asks next, so no CTA sits
// on a long tail of heavy tasks while others idle (the counter is caller
// scratch, cleared on the stream before each launch).
// Every wait is bounded (see ptx.cuh); on a timeout the CTA records the
// failing site in the status word, every role leaves its loop, in-flight
// copies and MMAs are drained with bounded waits and TMEM is freed.
//
// Build variants (template argument VAR, fixed-length and direct epilogue
// modes only; the default kernels compile none of this code):
//   VAR & kVarTrace    an event log: lane 0 of each role's first warp stamps
//                      clock64 at the hand-offs of the protocol (waits and
//                      arrivals only, so the softmax's instruction schedule
//                      between them is untouched) into a caller buffer (one
//                      track per role and CTA).
//   VAR & kVarStagger  an ablation: the two softmax warpgroups take turns
//                      for their exponentials ("FlashAttention-4 wiki", "Core
//                      methods": the staggered exp sections of S0 and S1).
//   VAR & kVarCheck  device-side checks: every decoded task, TMA coordinate,
//                    TMEM base and lane quadrant, shared-memory extent and
//                    epilogue store index is checked before use, and at exit
//                    the roles' counts of every hand-off (tiles loaded and
//                    consumed, S commits and waits, P arrivals and waits,
//                    O-done commits and waits) must agree.  A failed check
//                    records FA_ERR_DEVICE_CHECK and its site in the status
//                    word, skips the access and aborts the CTA like a timeout.
#pragma once
#include <cuda.h>

#include <type_traits>

#include "fa_schedule.h"
#include "ptx.cuh"

namespace fa {

constexpr int kThreads = 512;
// registers the setmaxnreg split needs: 128 x (176 + 176 + 104 + 56)
constexpr int kRegBudgetPerCta = 128 * (176 + 176 + 104 + 56);
constexpr int kChunkBytes = 128 * 64 * 2;  // 128 rows x 64 bf16: one 128B-swizzled TMA box
constexpr uint32_t kTmemCols = 512;
constexpr float kLn2 = 0.693147180559945309417f;
constexpr int kTaskRing = 4;     // task indices the TMA thread may post ahead (DYN)

// kernel modes
enum : int {
  kModeFixed = 0,
  kModeEmu = 1,
  kModeVarlen = 2,
  kModeDyn = 3,
  kModeSplit = 4,
  kModeDirect = 5,  // fixed-length, O rows stored straight from registers (short tasks)
  kNumModes = 6
};
constexpr int kTaskReaders = 13; // arrivals that free a ring slot: MMA warp + 12 softmax/correction warps

// debug_flags bits
constexpr int kDebugSkipPArrive = 1;  // softmax never arrives on p_full: exercises the bounded waits
constexpr int kDebugCountRescale = 2; // count the correction warps' O round trips in status word 3
constexpr int kDebugChecks = 4;       // run the checking instantiation (VAR & kVarCheck)
constexpr int kDebugPlantBadTask = 8; // checking instantiation: task 0 decodes to batch B (out of range)

// VAR template bits (build variants)
constexpr int kVarTrace = 1;
constexpr int kVarCheck = 2;
constexpr int kVarStagger = 4;

struct Params {
  CUtensorMap tm_q;  // 5-D view (d, pack, groups, Sq, B) of q (varlen: S = total_q rows, B = 1)
  CUtensorMap tm_k;  // 4-D view (d, Hkv, Sk, B) of k (varlen: S = total_k rows, B = 1)
  CUtensorMap tm_v;  // 4-D view (dv, Hkv, Sk, B) of v
  CUtensorMap tm_o;  // 5-D view (dv, pack, groups, Sq, B) of o
  float* lse;        // [B, Hq, Sq] (varlen: [Hq, total_q]) or null
  int64_t lse_bstride, lse_hstride;  // element strides of lse per batch and per head
  uint16_t* o;                       // o (bf16 bits): direct stores of ragged varlen tiles
  int64_t o_row_stride;              // elements between consecutive positions of o (Hq * dv)
  int o_align32;                     // o is 32-byte aligned: direct stores of 32 bytes
  const VarlenTask* vtasks;          // varlen: the planned task list
  const int* vtask_count;            // varlen: its length
  unsigned int* sched_next;          // DYN: next task index (cleared before the launch)
  float* opart;                      // split-KV: O / row_sum per range, [splits, B, Sq, Hq, dv]
  float* lpart;                      // split-KV: LSE per range, [splits, B, Hq, Sq]
  unsigned int* status;
  Problem prob;  // varlen: the shared fields (heads, pack, causal); lengths come per task
  float scale_log2;  // scale * log2(e)
  float tau;         // conditional-rescale threshold, log2 units
  unsigned long long timeout_ns;
  int debug_flags;
  uint64_t* trace;   // VAR & kVarTrace: [trace_ctas][kTraceTracks][1 + trace_cap] words
  int trace_ctas;    // CTAs 0 .. trace_ctas-1 record
  int trace_cap;     // records kept per track
};

template <int DQ, int DV>
struct Layout {
  static_assert(DQ % 64 == 0 && DV % 64 == 0 && DV <= DQ && DV <= 128 && DQ <= 192, "head dims");
  static constexpr int NQC = DQ / 64;  // 64-column chunks of a Q or K tile
  static constexpr int NVC = DV / 64;
  static constexpr int kQBytes = NQC * kChunkBytes;
  static constexpr int kSlotBytes = NQC * kChunkBytes;  // a ring slot holds one K tile or one V tile
  static constexpr int kStageOBytes = kChunkBytes;
  // [stage][acc_scale, (row_sum, ref) x task parity][row]: the final statistics
  // alternate between two slots so that a stage's last-block P V need not wait
  // for them to be read
  static constexpr int kMboxBytes = 2 * 5 * 128 * 4;
  static constexpr int kMaxSmem = 232448;              // 227 KB per CTA (opt-in)
  static constexpr int kFixed = 2 * kQBytes + kStageOBytes + kMboxBytes + 1024 + 1024;
  static constexpr int NS_fit = (kMaxSmem - kFixed) / kSlotBytes;
  static constexpr int NS = NS_fit > 8 ? 8 : NS_fit;  // K/V ring depth (tiles)
  static_assert(NS >= 2, "K/V ring needs two slots");

  static constexpr int oQ = 0;
  static constexpr int oRing = oQ + 2 * kQBytes;
  static constexpr int oStage = oRing + NS * kSlotBytes;
  static constexpr int oMbox = oStage + kStageOBytes;
  static constexpr int oBar = oMbox + kMboxBytes;

  // barrier indices
  static constexpr int bQFull = 0;        // [2]
  static constexpr int bQEmpty = 2;       // [2]
  static constexpr int bKvFull = 4;       // [NS]
  static constexpr int bKvEmpty = 4 + NS; // [NS]
  static constexpr int bSFull = 4 + 2 * NS;
  static constexpr int bPFull = bSFull + 2;
  static constexpr int bODone = bPFull + 2;
  static constexpr int bCorrFull = bODone + 2;
  static constexpr int bFinFull = bCorrFull + 2;  // [stage][task parity] final row_sum / reference posted (count 128)
  static constexpr int bStagger = bFinFull + 4;   // [2] (VAR & kVarStagger) stage s finished its exps (count 128)
  static constexpr int bEpiFull = bStagger + 2;   // WG2: staging tile written (count 128)
  static constexpr int bStageFree = bEpiFull + 1; // WG2: TMA store finished reading staging (count 1)
  static constexpr int bDrain = bStageFree + 1;   // MMA drain at exit
  static constexpr int bSink = bDrain + 1;      // arrivals nobody waits for (count 256)
  static constexpr int bTaskFull = bSink + 1;                // [kTaskRing] (DYN) count 1
  static constexpr int bTaskEmpty = bTaskFull + kTaskRing;   // [kTaskRing] (DYN) count kTaskReaders
  static constexpr int kNumBars = bTaskEmpty + kTaskRing;

  static constexpr int oMisc = oBar + kNumBars * 8;  // [0] TMEM base, [1] abort flag
  static constexpr int oTaskRing = oMisc + 16;       // int[kTaskRing] (DYN)
  static constexpr int oDbgCount = oTaskRing + 4 * kTaskRing;  // uint32[kDbgCounts] (VAR & kVarCheck)
  static constexpr int kBytes = oDbgCount + 4 * 24;
  static constexpr int kDynSmem = kBytes + 1024;     // slack to align the base to 1024 B
  static_assert(kDynSmem <= kMaxSmem, "shared memory budget");
};

// Wait-site codes recorded in status[1] on a timeout: role * 100 + barrier.
enum : unsigned int {
  kSiteSoftmaxS = 101,
  kSiteSoftmaxTask = 102,
  kSiteSoftmaxStagger = 103,
  kSiteCorrCorr = 201,
  kSiteCorrODone = 202,
  kSiteCorrEpiFull = 203,
  kSiteCorrStageFree = 204,
  kSiteCorrFin = 205,
  kSiteCorrTask = 206,
  kSiteMmaKv = 301,
  kSiteMmaQ = 302,
  kSiteMmaP = 303,
  kSiteMmaDrain = 304,
  kSiteMmaTask = 305,
  kSiteLoadQ = 401,
  kSiteLoadKv = 402,
  kSiteLoadDrain = 403,
  kSiteLoadTask = 404,
};

// The tasks a CTA walks: decoded from the fixed-length problem, or read from
// the list the varlen planning kernel wrote (every role reads the same list).
// An int the compiler cannot see through (keeps a re-read from being merged
// with an earlier one, so the earlier value need not stay live).
__device__ __forceinline__ int opaque_i32(int x) {
  asm volatile("" : "+r"(x));
  return x;
}
template <bool VARLEN>
__device__ __forceinline__ int task_count(const Params& p) {
  if constexpr (VARLEN) return *p.vtask_count;
  else return static_cast<int>(p.prob.num_tasks);
}

// FD: decode with the FastDiv fields (short-task kernels, where the decoding
// sits on the path between tasks); the causal kernels always do (their paired
// order takes several divisions per task, and a run-time division is a
// reciprocal on the SFU, queued behind the softmax's exponentials); the
// non-causal long-task kernels divide plainly.  BAL: the balanced static
// orders (key-split last wave without the mask, paired order with it) may be
// in use; dynamically scheduled kernels leave them out.
template <bool VARLEN, bool SPLIT, bool CAUSAL, bool FD, bool BAL>
__device__ __forceinline__ Task get_task(const Params& p, int t) {
  if constexpr (SPLIT) {
    return decode_split_task(p.prob, t);
  } else if constexpr (VARLEN) {
    const int4* r = reinterpret_cast<const int4*>(p.vtasks + t);
    const int4 a = r[0], b = r[1];
    VarlenTask rec;
    rec.b = a.x, rec.g = a.y, rec.mb = a.z, rec.reserved = a.w;
    rec.q_row0 = b.x, rec.sq = b.y, rec.k_row0 = b.z, rec.sk = b.w;
    return task_from_record(p.prob, rec);
  } else {
    if constexpr (FD) return decode_task_k<CAUSAL ? 1 : 0, true, BAL && !CAUSAL, BAL && CAUSAL>(p.prob, t);
    else if constexpr (CAUSAL) return decode_task_k<1, true, false, BAL>(p.prob, t);
    else return decode_task_k<-1, false, BAL, false>(p.prob, t);
  }
}

// Task k of this CTA for a reading warp (softmax, correction, MMA): the
// static index, or (DYN) the index the TMA thread posted in ring slot
// k % kTaskRing.  Returns -1 when no task is left, -2 on an abort.  Called by
// every lane of the warp.
template <int DQ, int DV, bool DYN>
__device__ __forceinline__ int read_task(int k, int num_tasks, uint32_t bar0, const volatile int* ring,
                                         const WaitCtx& wc, unsigned site) {
  using L = Layout<DQ, DV>;
  if constexpr (!DYN) {
    const int t = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
    return t < num_tasks ? t : -1;
  } else {
    const int slot = k % kTaskRing;
    const uint32_t parity = static_cast<uint32_t>(k / kTaskRing) & 1u;
    if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8u * (L::bTaskFull + slot), parity, wc, site))) return -2;
    const int t = ring[slot];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar0 + 8u * (L::bTaskEmpty + slot));
    return t;
  }
}

// The TMA thread's side (DYN): take the next task index from the global
// counter and post it in ring slot k % kTaskRing once every reader freed the
// slot's previous use.  Returns the index, -1 when none is left, -2 on an
// abort.  Static assignment needs no posting.
template <int DQ, int DV, bool DYN>
__device__ __forceinline__ int post_task(const Params& p, int k, int num_tasks, uint32_t bar0, volatile int* ring,
                                         const WaitCtx& wc) {
  using L = Layout<DQ, DV>;
  if constexpr (!DYN) {
    const int t = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
    return t < num_tasks ? t : -1;
  } else {
    const int slot = k % kTaskRing;
    if (k >= kTaskRing &&
        !mbar_wait(bar0 + 8u * (L::bTaskEmpty + slot), static_cast<uint32_t>(k / kTaskRing - 1) & 1u, wc,
                   kSiteLoadTask))
      return -2;
    const unsigned int got = atomicAdd(p.sched_next, 1u);
    const int t = got < static_cast<unsigned int>(num_tasks) ? static_cast<int>(got) : -1;
    ring[slot] = t;
    mbar_arrive(bar0 + 8u * (L::bTaskFull + slot));
    return t;
  }
}

// A wait that ignores the abort flag (used to drain in-flight async work
// before TMEM is freed); still bounded by the time limit.
__device__ __forceinline__ void mbar_drain_wait(uint32_t bar, uint32_t parity, const WaitCtx& w, unsigned site) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > w.timeout_ns) {
      raise_abort(w, kStatusTimeout, site);
      return;
    }
  }
}

// ---------------------------------------------------------------------------
// debug instantiations: the event log and the checks
// ---------------------------------------------------------------------------
// Event log: track = role (softmax stage 0, softmax stage 1, correction, MMA,
// TMA; in the backward: row warps of stage 0 and 1, unused, MMA, TMA); a
// record is one 64-bit word {code (bits 56-63), argument (bits 32-55),
// clock64 low 32 bits}.  Word 0 of a track holds its record count (records
// past trace_cap are counted, not kept).
constexpr int kTraceTracks = 5;
enum : uint32_t {
  // softmax (argument: block j; task: task index)
  kEvSmTask = 1, kEvSmWait = 2, kEvSmS = 3, kEvSmLd = 4, kEvSmMax = 5, kEvSmExp0 = 6, kEvSmExp1 = 7, kEvSmP = 8,
  // correction (argument: stage << 16 | block, or stage)
  kEvCoTask = 16, kEvCoCorr = 17, kEvCoRescaled = 18, kEvCoArrive = 19, kEvCoODone = 20, kEvCoEpi = 21,
  // MMA (argument: ring tile, stage, or stage << 16 | block)
  kEvMmTask = 32, kEvMmKv = 33, kEvMmQ = 34, kEvMmP = 35, kEvMmPV = 36, kEvMmQK = 37,
  // TMA (argument: stage or ring tile)
  kEvLdTask = 48, kEvLdQ = 49, kEvLdKvWait = 50, kEvLdKv = 51,
  // backward, row warps of stage s (tracks 0 / 1; argument: streamed block of the task, or task)
  kEvBrTask = 64, kEvBrWait = 65, kEvBrS = 66, kEvBrP = 67, kEvBrAcc = 68, kEvBrEpi = 69,
  // backward, MMA warp (track 3; argument: stage << 16 | block, or task)
  kEvBmTask = 80, kEvBmP = 81, kEvBmAcc = 82, kEvBmT = 83, kEvBmSdp = 84,
  // backward, TMA thread (track 4; argument: half-tile index, or task)
  kEvBlTask = 96, kEvBlT = 97,
};

// Keeps two registers per recording role (the record count and the on
// flag; a third for the track when TRACK < 0, i.e. chosen at run time): the
// track's address is recomputed from the kernel parameters, which live in
// parameter space, at each record.  PARAMS is the forward's Params or the
// backward's BwdParams (both carry trace, trace_ctas and trace_cap).
template <bool ON, int TRACK>
struct Tracer {
  uint32_t n = 0;
  bool on = false;
  int track = TRACK;
  template <class PARAMS>
  __device__ __forceinline__ void init(const PARAMS& p, bool recorder, int trk = TRACK) {
    if constexpr (ON) {
      on = recorder && p.trace != nullptr && static_cast<int>(blockIdx.x) < p.trace_ctas;
      if constexpr (TRACK < 0) track = trk;
    }
  }
  template <class PARAMS>
  __device__ __forceinline__ uint64_t* base(const PARAMS& p) const {
    const int tr = TRACK < 0 ? track : TRACK;
    return p.trace + (static_cast<int64_t>(blockIdx.x) * kTraceTracks + tr) * (p.trace_cap + 1);
  }
  template <class PARAMS>
  __device__ __forceinline__ void ev(const PARAMS& p, uint32_t code, uint32_t arg) {
    if constexpr (ON) {
      if (on) {
        if (n < static_cast<uint32_t>(p.trace_cap))
          base(p)[1 + n] = (static_cast<uint64_t>(code) << 56) | (static_cast<uint64_t>(arg & 0xFFFFFFu) << 32) |
                           static_cast<uint32_t>(clock64());
        ++n;
      }
    }
  }
  template <class PARAMS>
  __device__ __forceinline__ void finish(const PARAMS& p) {
    if constexpr (ON) {
      if (on) base(p)[0] = n;
    }
  }
};

// Hand-off counts each role keeps in the checking build (slots of the shared
// counter area, written by one lane at exit and compared by thread 0).
enum : int {
  kCntLdKv = 0, kCntLdQ = 1,                   // [2]: tiles / Q tiles loaded
  kCntMmKv = 3, kCntMmQ = 4,                   // [2]: tiles / Q tiles consumed
  kCntMmS = 6, kCntMmP = 8, kCntMmODone = 10,  // [2] each: S commits, P waits, O-done commits
  kCntSmS = 12, kCntSmP = 14,                  // [2] each: S waits, P arrivals
  kCntCoCorr = 16, kCntCoP = 18, kCntCoODone = 20,  // [2] each
  kNumCounts = 22
};
static_assert(kNumCounts <= 24, "counter area");

template <bool ON>
struct Counts {
  uint32_t c[ON ? kNumCounts : 1] = {};
  __device__ __forceinline__ void inc(int i) {
    if constexpr (ON) ++c[i];
  }
  __device__ __forceinline__ void add(int i, uint32_t v) {
    if constexpr (ON) c[i] += v;
  }
  // store slots [lo, hi) (one lane)
  __device__ __forceinline__ void store(uint32_t* area, int lo, int hi, bool writer) const {
    if constexpr (ON) {
      if (writer)
        for (int i = lo; i < hi; ++i) area[i] = c[i];
    }
  }
};

// Check sites recorded with FA_ERR_DEVICE_CHECK
enum : unsigned int {
  kSiteCheckTask = 701,      // a decoded task outside the problem
  kSiteCheckQCoord = 702,    // a Q tile coordinate outside the tensor
  kSiteCheckKvCoord = 703,   // a K/V tile coordinate outside the tensor
  kSiteCheckSmem = 704,      // the shared-memory layout past the launch's dynamic size
  kSiteCheckTmem = 705,      // TMEM base not at lane 0 / column 0, or a lane quadrant off its warp
  kSiteCheckOStore = 706,    // an output row or tile outside O
  kSiteCheckLse = 707,       // an LSE index outside lse
  kSiteCheckCounts = 710,    // + i: the i-th hand-off count comparison failed
};

__device__ __forceinline__ bool dbg_check(bool ok, const WaitCtx& wc, unsigned site) {
  if (!ok) raise_abort(wc, kStatusCheck, site);
  return ok;
}

// Is a decoded fixed-length task inside the problem?
__device__ __forceinline__ bool task_in_problem(const Problem& pr, const Task& tk) {
  const int kb = (tk.kend + kBN - 1) / kBN;
  bool ok = tk.bc >= 0 && tk.bc < pr.B && tk.g >= 0 && tk.g < pr.groups && tk.kvh >= 0 && tk.kvh < pr.Hkv &&
            tk.q_row0 >= 0 && tk.k_row0 >= 0 && tk.nmax == max(tk.n[0], tk.n[1]) && tk.sq == pr.Sq;
#pragma unroll
  for (int s = 0; s < 2; ++s)
    ok = ok && tk.n[s] >= 0 && tk.n[s] <= kb && tk.pos0[s] >= 0 && (tk.n[s] == 0 || tk.pos0[s] < tk.sq);
  if (tk.ksplit != 0) ok = ok && tk.ksplit == tk.n[0] && tk.n[0] + tk.n[1] <= kb;
  return ok;
}

// The checking build's view of a decoded task: the planted fault (debug
// flag), then the range check.  Warp-uniform (every lane decodes the same
// task).  Returns false after recording the failure.
template <bool CK>
__device__ __forceinline__ bool check_task(const Params& p, Task& tk, int task, const WaitCtx& wc) {
  if constexpr (CK) {
    if ((p.debug_flags & kDebugPlantBadTask) && task == 0) tk.bc = p.prob.B;
    return dbg_check(task_in_problem(p.prob, tk), wc, kSiteCheckTask);
  } else {
    return true;
  }
}

// ---------------------------------------------------------------------------
// 2^x on the FMA pipe ("FlashAttention-4 wiki", "Core methods": Cody-Waite
// range reduction and a degree-3 Horner polynomial, the integer part added to
// the exponent field).  x = j + f with j = rint(x) (adding 1.5 * 2^23 rounds
// to an integer and leaves j in the low mantissa bits), f in [-1/2, 1/2];
// 2^f from a polynomial fitted by exp2_poly.py (max relative error 7.5e-5,
// below half a bf16 unit).  x is clamped at -126 so the exponent sum stays in
// range; only unmasked blocks use it (a masked key must give exactly 0).
// ---------------------------------------------------------------------------
constexpr float kExp2C0 = 0.99992806f;
constexpr float kExp2C1 = 0.69326097f;
constexpr float kExp2C2 = 0.24261114f;
constexpr float kExp2C3 = 0.055171628f;

__device__ __forceinline__ void ex2_fma_x2(uint64_t x2, float& y0, float& y1) {
  float a, b;
  f2_unpack(x2, a, b);
  const uint64_t xc = f2_pack(fmaxf(a, -126.f), fmaxf(b, -126.f));
  const uint64_t t = f2_add(xc, f2_pack(12582912.f, 12582912.f));    // 1.5 * 2^23 + rint(x)
  const uint64_t jf = f2_add(t, f2_pack(-12582912.f, -12582912.f));  // rint(x)
  const uint64_t f = f2_fma(jf, f2_pack(-1.f, -1.f), xc);            // x - rint(x)
  uint64_t q = f2_fma(f2_pack(kExp2C3, kExp2C3), f, f2_pack(kExp2C2, kExp2C2));
  q = f2_fma(q, f, f2_pack(kExp2C1, kExp2C1));
  q = f2_fma(q, f, f2_pack(kExp2C0, kExp2C0));
  float t0, t1, q0, q1;
  f2_unpack(t, t0, t1);
  f2_unpack(q, q0, q1);
  // the low bits of t hold rint(x); shifted by 23 they add to the exponent
  y0 = __uint_as_float(__float_as_uint(q0) + (__float_as_uint(t0) << 23));
  y1 = __uint_as_float(__float_as_uint(q1) + (__float_as_uint(t1) << 23));
}

// ---------------------------------------------------------------------------
// softmax (WG0 / WG1)
// ---------------------------------------------------------------------------
// EMU: one in four exponentials of unmasked blocks on the FMA pipe (an option;
// its own instantiation, so the default kernel carries no extra code)
template <int DQ, int DV, bool CAUSAL, bool EMU, bool VARLEN, bool DYN, bool SPLIT, bool FD, int VAR>
__device__ __forceinline__ void softmax_role(const Params& p, const int stage, const uint32_t tmem,
                                             const uint32_t sbase, float* mbox, const volatile int* ring,
                                             uint32_t* dbg_area, const WaitCtx& wc) {
  using L = Layout<DQ, DV>;
  constexpr bool CK = (VAR & kVarCheck) != 0;
  const Problem& pr = p.prob;
  const int t = threadIdx.x - stage * 128;  // row of the Q tile == TMEM lane
  const uint32_t tS = tmem + (static_cast<uint32_t>(t & ~31) << 16) + static_cast<uint32_t>(stage * 128);
  const uint32_t bar_s = sbase + L::oBar + 8 * (L::bSFull + stage);
  const uint32_t bar_corr = sbase + L::oBar + 8 * (L::bCorrFull + stage);
  const uint32_t bar_sink = sbase + L::oBar + 8 * L::bSink;
  const uint32_t bar_p = sbase + L::oBar + 8 * (L::bPFull + stage);
  const uint32_t bar_fin = sbase + L::oBar + 8 * (L::bFinFull + 2 * stage);  // [task parity]
  constexpr bool STAG = (VAR & kVarStagger) != 0;
  uint32_t stag_k = 0;  // staggered blocks of this stage so far (STAG)
  float* mb_acc = mbox + (stage * 5 + 0) * 128;
  float* mb_fin = mbox + (stage * 5 + 1) * 128;  // [task parity][row_sum, ref][row]
  const float sl2 = p.scale_log2;
  const float neg_tau = -p.tau;
  const bool skip_p = (p.debug_flags & kDebugSkipPArrive) != 0;
  // bit 0: phase of the S barrier; bit 1: parity of the tasks with blocks of
  // this stage so far (the slot of the final statistics).  One register.
  uint32_t phase = 0;
  const int num_tasks = task_count<VARLEN>(p);
  Tracer<(VAR & kVarTrace) != 0, -1> tr;  // track = stage
  tr.init(p, t == 0, stage);
  Counts<CK> cnt;
  if constexpr (CK) {  // this warp's TMEM lane quadrant is (warp % 4)
    if (!dbg_check((t & ~31) == 32 * ((threadIdx.x >> 5) & 3), wc, kSiteCheckTmem)) return;
  }

  for (int kt = 0;; ++kt) {
    const int task = read_task<DQ, DV, DYN>(kt, num_tasks, sbase + L::oBar, ring, wc, kSiteSoftmaxTask);
    if (task < 0) break;  // no task left, or an abort
    Task tk = get_task<VARLEN, SPLIT, CAUSAL, FD, !DYN>(p, task);
    if (!check_task<CK>(p, tk, task, wc)) break;
    tr.ev(p, kEvSmTask, static_cast<uint32_t>(task));
    const int n = stage ? tk.n[1] : tk.n[0];
    if (n == 0) continue;
    const int pos0 = stage ? tk.pos0[1] : tk.pos0[0];
    // keys of this stage counted from its first key: a key-split task's stage
    // 1 starts at block ksplit (non-causal only; 0 otherwise)
    const int kend = tk.kend - (CAUSAL ? 0 : stage * tk.ksplit * kBN);
    // last key visible to this row (inclusive, counted from the task's first
    // key; keys >= kend are never visible; pos + kshift stays inside 32 bits
    // for the sizes the host accepts; below -1 it means the same as -1), and
    // the first block that needs the element mask
    int last_key = kend - 1;
    if (CAUSAL) {
      const int c = pos0 + (FD ? fdiv(t, pr.fd_pack) : t / pr.pack) + tk.kshift;
      if (c < last_key) last_key = c;
    }
    if (last_key < -1) last_key = -1;
    const int j_mask = first_masked_block(kend, tk.kshift, CAUSAL, pos0);
    float row_max = -INFINITY;  // kept reference, raw score units
    float row_sum = 0.f;
    float ref = 0.f;            // row_max * scale_log2 (0 while the row is empty)

    for (int j = 0; j < n; ++j) {
      tr.ev(p, kEvSmWait, static_cast<uint32_t>(j));
      const bool ok = __all_sync(0xffffffffu, mbar_wait(bar_s, phase & 1u, wc, kSiteSoftmaxS));
      if (!ok) {
        tr.finish(p);
        return;
      }
      phase ^= 1u;
      cnt.inc(kCntSmS + stage);
      tc_fence_after();
      tr.ev(p, kEvSmS, static_cast<uint32_t>(j));

      uint32_t r[128];
      tmem_ld128_wait(tS, r);
      float s[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(r[c]);

      const bool masked_block = j >= j_mask;
      if (masked_block) {
        // columns c <= lim are visible
        const int lim = max(-1, min(127, last_key - j * kBN));
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > lim) s[c] = -INFINITY;
      }

      // block maximum: three-input max, four independent chains
      float m0 = fmaxf(s[0], s[1]), m1 = fmaxf(s[2], s[3]), m2 = fmaxf(s[4], s[5]), m3 = fmaxf(s[6], s[7]);
#pragma unroll
      for (int c = 8; c < 128; c += 8) {
        m0 = fmax3(m0, s[c + 0], s[c + 1]);
        m1 = fmax3(m1, s[c + 2], s[c + 3]);
        m2 = fmax3(m2, s[c + 4], s[c + 5]);
        m3 = fmax3(m3, s[c + 6], s[c + 7]);
      }
      const float bmax = fmaxf(fmax3(m0, m1, m2), m3);

      // conditional rescaling: keep the reference unless the maximum grew by
      // more than tau (log2 units); the first visible block takes its own max
      float acc = 1.f;
      if (bmax != -INFINITY) {
        if (row_max == -INFINITY) {
          row_max = bmax;
        } else if (bmax > row_max) {
          const float delta = (row_max - bmax) * sl2;
          if (delta < neg_tau) {
            acc = ex2_approx(delta);
            row_max = bmax;
          }
        }
      }
      ref = (row_max == -INFINITY) ? 0.f : row_max * sl2;

      // post acc_scale now: the correction warps rescale O (when needed) while
      // the exponentials below run, off the path to the PV MMA.  A first block
      // is not posted (its acc_scale is 1 and its P V writes O afresh; the
      // correction warps read the slot from the second block on): its arrival
      // goes to a barrier nobody waits for, chosen without a branch.
      mb_acc[t] = acc;
      mbar_arrive(j > 0 ? bar_corr : bar_sink);

      // p = 2^(s * scale_log2 - ref): one packed FMA per pair, then ex2; the
      // row sum is accumulated in packed pairs of fp32.  P goes to TMEM as
      // packed bf16 pairs, 64 keys at a time.
      const uint64_t sl2x2 = f2_pack(sl2, sl2);
      const uint64_t nrefx2 = f2_pack(-ref, -ref);
      uint64_t sum_a = f2_pack(0.f, 0.f), sum_b = sum_a;
      auto exps = [&](auto emu_tag) {
        constexpr bool kFma = decltype(emu_tag)::value;  // one pair in four on the FMA pipe
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int c = 64 * half; c < 64 * half + 64; c += 4) {
            float x0, x1, x2, x3;
            f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), sl2x2, nrefx2), x0, x1);
            s[c] = ex2_approx(x0);
            s[c + 1] = ex2_approx(x1);
            const uint64_t xb = f2_fma(f2_pack(s[c + 2], s[c + 3]), sl2x2, nrefx2);
            if (kFma && (c & 4)) {
              ex2_fma_x2(xb, s[c + 2], s[c + 3]);
            } else {
              f2_unpack(xb, x2, x3);
              s[c + 2] = ex2_approx(x2);
              s[c + 3] = ex2_approx(x3);
            }
            sum_a = f2_add(sum_a, f2_pack(s[c], s[c + 1]));
            sum_b = f2_add(sum_b, f2_pack(s[c + 2], s[c + 3]));
          }
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) pk[i] = pack_bf16x2(s[64 * half + 2 * i], s[64 * half + 2 * i + 1]);
          tmem_st32(tS + static_cast<uint32_t>(32 * half), pk);
        }
      };
      // staggered exponential sections (ablation): in the blocks both stages
      // visit, stage 1 starts its exponentials after stage 0 finished those of
      // the same block, and stage 0 after stage 1 finished those of the
      // previous such block
      const bool staggered = STAG && j < min(tk.n[0], tk.n[1]);
      if constexpr (STAG) {
        if (staggered && (stage == 1 || stag_k > 0)) {
          const uint32_t other = sbase + L::oBar + 8 * (L::bStagger + (stage ^ 1));
          const uint32_t par = (stage == 1 ? stag_k : stag_k - 1u) & 1u;
          if (!__all_sync(0xffffffffu, mbar_wait(other, par, wc, kSiteSoftmaxStagger))) {
            tr.finish(p);
            return;
          }
        }
      }
      if constexpr (EMU) {
        if (!masked_block) exps(std::true_type{});
        else exps(std::false_type{});
      } else {
        exps(std::false_type{});
      }
      if constexpr (STAG) {
        if (staggered) {
          mbar_arrive(sbase + L::oBar + 8 * (L::bStagger + stage));
          ++stag_k;
        }
      }
      tmem_wait_st();
      // P is in TMEM: signal the MMA warp first, then the row sum
      tc_fence_before();
      if (!skip_p) {
        mbar_arrive(bar_p);
        cnt.inc(kCntSmP + stage);
      }
      tr.ev(p, kEvSmP, static_cast<uint32_t>(j));
      float sa0, sa1;
      f2_unpack(f2_add(sum_a, sum_b), sa0, sa1);
      row_sum = row_sum * acc + (sa0 + sa1);
      if (j == n - 1) {  // final statistics for the epilogue, in this task's slot
        const uint32_t par = (phase >> 1) & 1u;
        mb_fin[(2 * par) * 128 + t] = row_sum;
        mb_fin[(2 * par + 1) * 128 + t] = ref;
        mbar_arrive(bar_fin + 8 * par);
        phase ^= 2u;
      }
    }
  }
  tr.finish(p);
  if (!*wc.abort_flag) {
    cnt.store(dbg_area, kCntSmS + stage, kCntSmS + stage + 1, t == 0);
    cnt.store(dbg_area, kCntSmP + stage, kCntSmP + stage + 1, t == 0);
  }
}

// ---------------------------------------------------------------------------
// correction + epilogue (WG2)
// ---------------------------------------------------------------------------
// COUNT: the FMA-exp2 ablation kernel and the checking build also count O
// rescales (debug_flags bit 1); the rescale decisions do not depend on how the
// exponentials are taken, and the default kernels carry no counting code.
template <int DQ, int DV, bool CAUSAL, bool VARLEN, bool DYN, bool SPLIT, bool DIRECT, bool COUNT, int VAR>
__device__ __forceinline__ void correction_role(const Params& p, const uint32_t tmem, const uint32_t sbase,
                                                uint8_t* smem, float* mbox, const volatile int* ring,
                                                uint32_t* dbg_area, const WaitCtx& wc) {
  using L = Layout<DQ, DV>;
  constexpr bool CK = (VAR & kVarCheck) != 0;
  constexpr bool TS = !CAUSAL && !VARLEN && !DYN && !SPLIT;  // key-split tail tasks possible
  const Problem& pr = p.prob;
  const int t = threadIdx.x - 256;  // row == TMEM lane
  const uint32_t lane_off = static_cast<uint32_t>(t & ~31) << 16;
  const uint32_t bar0 = sbase + L::oBar;
  uint8_t* staging = smem + L::oStage;
  const uint32_t staging_s = sbase + L::oStage;
  uint32_t corr_phase[2] = {0u, 0u};
  uint32_t fin_k[2] = {0u, 0u};     // final statistics read (one per task with blocks; slot = parity)
  uint32_t od_count[2] = {0u, 0u};  // o_done phases consumed (one per task with blocks)
  uint32_t chunks = 0;              // epilogue chunks stored through the staging tile so far
  const int num_tasks = task_count<VARLEN>(p);
  // short-task kernels with static assignment: the next task is decoded
  // before the current task's epilogue (while the last P V run), so that the
  // next task's first hand-off does not wait behind the decoding
  constexpr bool kPre = DIRECT && !DYN;
  Task nxt{};
  Tracer<(VAR & kVarTrace) != 0, 2> tr;
  tr.init(p, t == 0);
  Counts<CK> cnt;
  // The P-ready barrier of a stage's first block in a task also says that O is
  // free: these warps arrive on it as soon as the previous task's epilogue has
  // read the stage's O out of TMEM (here: before the first task), not when the
  // block comes up, so that the next task's first P V need not wait behind the
  // other stage's epilogue.
  auto o_free = [&](int s) {
    tc_fence_before();
    mbar_arrive(bar0 + 8 * (L::bPFull + s));
    tr.ev(p, kEvCoArrive, static_cast<uint32_t>(s << 16));
  };
  // the final row sum and reference of stage s in the current task (the
  // softmax alternates between two slots by task parity)
  auto read_fin = [&](int s, float& sum, float& ref) -> bool {
    const uint32_t par = fin_k[s] & 1u;
    if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * (L::bFinFull + 2 * s + static_cast<int>(par)),
                                           (fin_k[s] >> 1) & 1u, wc, kSiteCorrFin)))
      return false;
    ++fin_k[s];
    sum = mbox[(s * 5 + 1 + 2 * static_cast<int>(par)) * 128 + t];
    ref = mbox[(s * 5 + 2 + 2 * static_cast<int>(par)) * 128 + t];
    return true;
  };
  if constexpr (CK) {  // this warp's TMEM lane quadrant is (warp % 4)
    if (!__all_sync(0xffffffffu, dbg_check((t & ~31) == 32 * ((threadIdx.x >> 5) & 3), wc, kSiteCheckTmem)))
      goto out;
  }
  o_free(0);
  o_free(1);
  if constexpr (kPre) {
    const int t0 = read_task<DQ, DV, DYN>(0, num_tasks, bar0, ring, wc, kSiteCorrTask);
    if (t0 >= 0) nxt = get_task<VARLEN, SPLIT, CAUSAL, DIRECT, !DYN>(p, t0);
  }
  for (int kt = 0;; ++kt) {
    const int task = read_task<DQ, DV, DYN>(kt, num_tasks, bar0, ring, wc, kSiteCorrTask);
    if (task < 0) break;  // no task left, or an abort
    Task tk = kPre ? nxt : get_task<VARLEN, SPLIT, CAUSAL, DIRECT, !DYN>(p, task);
    if (!check_task<CK>(p, tk, task, wc)) break;
    tr.ev(p, kEvCoTask, static_cast<uint32_t>(task));
    float fin_sum[2] = {0.f, 0.f}, fin_ref[2] = {0.f, 0.f};

    // first blocks: nothing to rescale, and their P-ready arrival was made
    // when O became free
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      if (tk.n[s] > 0) {
        cnt.inc(kCntCoCorr + s);
        cnt.inc(kCntCoP + s);
      }
    }
    for (int j = 1; j < tk.nmax; ++j) {
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        if (j >= tk.n[s]) continue;
        const bool ok = __all_sync(0xffffffffu,
                                   mbar_wait(bar0 + 8 * (L::bCorrFull + s), corr_phase[s], wc, kSiteCorrCorr));
        if (!ok) goto out;
        corr_phase[s] ^= 1u;
        cnt.inc(kCntCoCorr + s);
        tr.ev(p, kEvCoCorr, static_cast<uint32_t>(s << 16 | j));
        const float acc = mbox[(s * 5 + 0) * 128 + t];
        // warp-uniform skip of the O round trip when no row moved its
        // reference.  The softmax posted acc_scale after S_j was ready, and S_j
        // ready implies that P V_{j-1} completed, so O is final here.
        if (__any_sync(0xffffffffu, acc != 1.f)) {
          if constexpr (COUNT) {
            if ((p.debug_flags & kDebugCountRescale) && (t & 31) == 0) atomicAdd(p.status + 3, 1u);
          }
          tc_fence_after();
          const uint32_t tO = tmem + lane_off + 256u + static_cast<uint32_t>(s * 128);
#pragma unroll
          for (int c = 0; c < DV; c += 32) {
            uint32_t r[32];
            tmem_ld32_wait(tO + c, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * acc);
            tmem_st32(tO + c, r);
          }
          tmem_wait_st();
          tr.ev(p, kEvCoRescaled, static_cast<uint32_t>(s << 16 | j));
        }
        tc_fence_before();
        mbar_arrive(bar0 + 8 * (L::bPFull + s));
        cnt.inc(kCntCoP + s);
        tr.ev(p, kEvCoArrive, static_cast<uint32_t>(s << 16 | j));
      }
    }

    // epilogue: O / row_sum -> bf16 -> staging -> TMA store; LSE.  A varlen
    // task record is read again here rather than kept in registers across
    // the K/V loop (this role runs at 104 registers).
    if constexpr (VARLEN) tk = get_task<VARLEN, false, CAUSAL, false, false>(p, opaque_i32(task));
    if constexpr (kPre) {
      const int t1 = read_task<DQ, DV, DYN>(kt + 1, num_tasks, bar0, ring, wc, kSiteCorrTask);
      if (t1 >= 0) nxt = get_task<VARLEN, SPLIT, CAUSAL, DIRECT, !DYN>(p, t1);
    }
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      // key-split tail task: one output tile, both halves merged at s = 0
      const bool merge = TS && tk.ksplit != 0;
      if (merge && s == 1) continue;
      const int pos0 = tk.pos0[s];
      if (pos0 >= tk.sq) continue;  // tile past the end of the sequence
      const bool has = tk.n[s] > 0;
      // rows stored one by one from registers in the direct-epilogue mode and
      // for variable-length batches (their tasks are mostly short, and a TMA
      // store of a tile that runs past its sequence would write the next
      // sequence's rows; measured on varlen32k: +5 % over staged TMA stores)
      const bool direct = DIRECT || VARLEN;
      const int row_pos = DIRECT ? fdiv(t, pr.fd_pack) : t / pr.pack;
      const int pos = pos0 + row_pos;
      const int head = tk.g * pr.pack + (t - row_pos * pr.pack);
      if (has && !read_fin(s, fin_sum[s], fin_ref[s])) goto out;
      if (merge && !read_fin(1, fin_sum[1], fin_ref[1])) goto out;
      if (has) {  // o_done completes once per task: after the stage's last P V
        const bool ok =
            __all_sync(0xffffffffu, mbar_wait(bar0 + 8 * (L::bODone + s), od_count[s] & 1u, wc, kSiteCorrODone));
        if (!ok) goto out;
        ++od_count[s];
        tc_fence_after();
        tr.ev(p, kEvCoODone, static_cast<uint32_t>(s));
      }
      float inv = 0.f, lse = -INFINITY;
      float inv1 = 0.f;  // merge: weight of stage 1's O
      if (merge) {
        // the two key halves: reference m_s and row sum l_s each (log2
        // units); with m = max m_s, l = sum 2^(m_s - m) l_s, and
        // O = sum 2^(m_s - m) O_s / l, LSE = (m + log2 l) ln 2
        const bool ok =
            __all_sync(0xffffffffu, mbar_wait(bar0 + 8 * (L::bODone + 1), od_count[1] & 1u, wc, kSiteCorrODone));
        if (!ok) goto out;
        ++od_count[1];
        tc_fence_after();
        const float m0 = fin_sum[0] > 0.f ? fin_ref[0] : -INFINITY;
        const float m1 = fin_sum[1] > 0.f ? fin_ref[1] : -INFINITY;
        const float m = fmaxf(m0, m1);
        if (m != -INFINITY) {
          const float w0 = ex2_approx(m0 - m), w1 = ex2_approx(m1 - m);  // 2^-inf = 0
          const float l = w0 * fin_sum[0] + w1 * fin_sum[1];
          const float il = 1.f / l;
          inv = w0 * il;
          inv1 = w1 * il;
          lse = (m + __log2f(l)) * kLn2;
        }
      } else if (has && fin_sum[s] > 0.f) {
        inv = 1.f / fin_sum[s];
        lse = (fin_ref[s] + __log2f(fin_sum[s])) * kLn2;
      }
      const uint32_t tO = tmem + lane_off + 256u + static_cast<uint32_t>(s * 128);
      if constexpr (SPLIT) {
        // partial result of this key range: O / row_sum in fp32 and its LSE
        // (-inf, O = 0 when no key of the range is visible to the row).  The
        // TMEM loads are warp-collective: every lane runs them (has is
        // uniform); only the stores depend on the row.
        const bool store = pos < tk.sq;
        const int64_t row = ((static_cast<int64_t>(tk.split) * pr.B + tk.b) * pr.Sq + pos) * pr.Hq + head;
        float4* dst = reinterpret_cast<float4*>(p.opart + row * DV);
#pragma unroll 1
        for (int c = 0; c < DV; c += 32) {
          uint32_t r[32];
          if (has) {
            tmem_ld32_wait(tO + static_cast<uint32_t>(c), r);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
          }
          if (store) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[c / 4 + q] = make_float4(__uint_as_float(r[4 * q]) * inv, __uint_as_float(r[4 * q + 1]) * inv,
                                           __uint_as_float(r[4 * q + 2]) * inv, __uint_as_float(r[4 * q + 3]) * inv);
          }
        }
        if (has) o_free(s);
        if (store) p.lpart[((static_cast<int64_t>(tk.split) * pr.B + tk.b) * pr.Hq + head) * pr.Sq + pos] = lse;
        continue;
      }
      uint4* out_row = nullptr;
      if constexpr (CK) {  // the row this lane stores lies inside O
        const bool in_o = !direct || pos >= tk.sq ||
                          (static_cast<int64_t>(tk.bc) * tk.sq + tk.q_row0 + pos < static_cast<int64_t>(pr.B) * pr.Sq &&
                           head >= 0 && head < pr.Hq);
        if (!__all_sync(0xffffffffu, dbg_check(in_o, wc, kSiteCheckOStore))) goto out;
      }
      if (direct && pos < tk.sq)
        out_row = reinterpret_cast<uint4*>(p.o + (static_cast<int64_t>(tk.bc) * tk.sq + tk.q_row0 + pos) *
                                                     p.o_row_stride +
                                           static_cast<int64_t>(head) * DV);
#pragma unroll 1
      for (int c = 0; c < L::NVC; ++c) {
        if (!direct && chunks > 0) {
          const bool ok = __all_sync(0xffffffffu, mbar_wait(bar0 + 8 * L::bStageFree, (chunks - 1u) & 1u, wc,
                                                            kSiteCorrStageFree));
          if (!ok) goto out;
        }
        uint4* row = reinterpret_cast<uint4*>(staging + t * 128);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t r[32];
          float mul = inv;
          if (has) {
            tmem_ld32_wait(tO + static_cast<uint32_t>(c * 64 + half * 32), r);
            if (merge) {  // r = inv * O_0 + inv1 * O_1 (O_1 is 128 columns on)
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                uint32_t r1[16];
                tmem_ld16_wait(tO + static_cast<uint32_t>(128 + c * 64 + half * 32 + h * 16), r1);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  r[16 * h + i] = __float_as_uint(
                      fmaf(__uint_as_float(r1[i]), inv1, __uint_as_float(r[16 * h + i]) * inv));
              }
              mul = 1.f;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
          }
          uint4 v[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            v[q].x = pack_bf16x2(__uint_as_float(r[8 * q + 0]) * mul, __uint_as_float(r[8 * q + 1]) * mul);
            v[q].y = pack_bf16x2(__uint_as_float(r[8 * q + 2]) * mul, __uint_as_float(r[8 * q + 3]) * mul);
            v[q].z = pack_bf16x2(__uint_as_float(r[8 * q + 4]) * mul, __uint_as_float(r[8 * q + 5]) * mul);
            v[q].w = pack_bf16x2(__uint_as_float(r[8 * q + 6]) * mul, __uint_as_float(r[8 * q + 7]) * mul);
          }
          if (direct) {
            // a row's 64 bytes of this half: whole 32-byte sectors when O allows it
            if (out_row != nullptr) {
              uint4* dst = out_row + c * 8 + half * 4;
              if (p.o_align32) {
                st_global_v8(dst, v[0], v[1]);
                st_global_v8(dst + 2, v[2], v[3]);
              } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) dst[q] = v[q];
              }
            }
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) row[(half * 4 + q) ^ (t & 7)] = v[q];  // 128-byte swizzle of the TMA box
          }
        }
        if (c == L::NVC - 1) {  // the stage's O has been read out of TMEM
          if (has) o_free(s);
          if (merge) o_free(1);
        }
        if (direct) continue;
        fence_proxy_async_smem();
        mbar_arrive(bar0 + 8 * L::bEpiFull);
        bool stored = true;
        if (t == 0) {
          stored = mbar_wait(bar0 + 8 * L::bEpiFull, chunks & 1u, wc, kSiteCorrEpiFull);
          if constexpr (CK)  // the stored tile starts inside O
            stored = stored && dbg_check(tk.q_row0 + pos0 >= 0 && tk.q_row0 + pos0 < pr.Sq && tk.g >= 0 &&
                                             tk.g < pr.groups && tk.bc >= 0 && tk.bc < pr.B,
                                         wc, kSiteCheckOStore);
          if (stored) {
            tma_store_5d(&p.tm_o, staging_s, c * 64, 0, tk.g, tk.q_row0 + pos0, tk.bc);
            bulk_commit_group();
            bulk_wait_group_read0();
            mbar_arrive(bar0 + 8 * L::bStageFree);
          }
        }
        // the whole warp leaves together (its later collectives need every lane)
        stored = __all_sync(0xffffffffu, stored);
        ++chunks;
        if (!stored) goto out;
      }
      if (p.lse != nullptr && pos < tk.sq) {
        const int64_t li = tk.b * p.lse_bstride + head * p.lse_hstride + tk.q_row0 + pos;
        bool ok = true;
        if constexpr (CK) ok = dbg_check(li >= 0 && li < static_cast<int64_t>(pr.B) * pr.Hq * pr.Sq, wc, kSiteCheckLse);
        if (ok) p.lse[li] = lse;
      }
      tr.ev(p, kEvCoEpi, static_cast<uint32_t>(s));
    }
  }
out:
  if (t == 0) bulk_wait_group0();
  tr.finish(p);
  if (!*wc.abort_flag) {
    cnt.store(dbg_area, kCntCoCorr, kCntCoCorr + 2, t == 0);
    cnt.store(dbg_area, kCntCoP, kCntCoP + 2, t == 0);
    if constexpr (CK) {
      if (t == 0) {
        dbg_area[kCntCoODone] = od_count[0];
        dbg_area[kCntCoODone + 1] = od_count[1];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// MMA issue (warp 12, one thread)
// ---------------------------------------------------------------------------
// S = Q K^T: M = 128 rows, N = 128 keys, K = DQ in steps of 16 (32 bytes inside
// a 128-byte swizzled row; a new 16 KB chunk every 64 columns).  Descriptor
// start addresses are in 16-byte units, so offsets are added to the low field.
template <int DQ, int DV>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_addr, uint32_t k_addr, uint32_t leader) {
  constexpr uint32_t kIdesc = idesc_bf16_f32(128, 128, false, false);
#pragma unroll
  for (int c = 0; c < DQ / 64; ++c) {
    const uint32_t co = opaque_u32(static_cast<uint32_t>(c * kChunkBytes));
    mma_ss_x4<2, 2>(d_tmem, smem_desc_sw128(q_addr + co, 16, 1024), smem_desc_sw128(k_addr + co, 16, 1024), kIdesc,
                    c != 0 ? 1u : 0u, leader);
  }
}

// O (+)= P V for one half of the block (keys 64*half .. 64*half+63): M = 128
// rows, N = DV, K in steps of 16; P is read from TMEM (8 columns of packed bf16
// pairs per step), V from SMEM (MN-major: 16 key rows of 128 bytes per step;
// the second 64-column chunk of V is LBO away).
template <int DV>
__device__ __forceinline__ void issue_pv_half(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_addr, int half,
                                              bool accumulate, uint32_t leader) {
  constexpr uint32_t kIdesc = idesc_bf16_f32(128, DV, false, true);
  constexpr uint32_t kStep = 16 * 128 >> 4;  // 16 key rows, in 16-byte units
  const uint32_t va = opaque_u32(v_addr + static_cast<uint32_t>(half * 64 * 128));
  mma_ts_x4<kStep>(d_tmem, p_tmem + static_cast<uint32_t>(32 * half), smem_desc_sw128(va, kChunkBytes, 1024),
                   kIdesc, accumulate ? 1u : 0u, leader);
}

// K/V tiles are consumed in the order K0, V0, K1, V1, ...; a task starting
// at ring tile `base` has K_j at base + 2j and V_j at base + 2j + 1.
// o_done[s] is committed once per task, after the stage's last P V: inside a
// task, "S_j ready" already implies that P V_{j-1} has completed (a commit
// tracks every earlier MMA of the issuing thread).
template <int DQ, int DV, bool CAUSAL, bool VARLEN, bool DYN, bool SPLIT, bool FD, int VAR>
__device__ __forceinline__ void mma_role(const Params& p, const uint32_t tmem, const uint32_t sbase,
                                         const volatile int* ring, uint32_t* dbg_area, const WaitCtx& wc) {
  using L = Layout<DQ, DV>;
  constexpr bool CK = (VAR & kVarCheck) != 0;
  constexpr bool TS = !CAUSAL && !VARLEN && !DYN && !SPLIT;  // key-split tail tasks possible
  const uint32_t bar0 = sbase + L::oBar;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  auto slot_addr = [&](uint32_t it) { return sbase + L::oRing + (it % L::NS) * L::kSlotBytes; };
  auto q_addr = [&](int s) { return sbase + L::oQ + static_cast<uint32_t>(s * L::kQBytes); };
  uint32_t q_phase[2] = {0u, 0u}, p_phase[2] = {0u, 0u};
  uint32_t kv_it = 0;  // first ring tile of the current task
  constexpr bool kEarlyV = L::NS <= 3;
  const uint32_t leader = (threadIdx.x & 31) == 0 ? 1u : 0u;  // the lane that issues MMAs and commits
  Tracer<(VAR & kVarTrace) != 0, 3> tr;
  tr.init(p, leader != 0);
  Counts<CK> cnt;
  // every lane waits; a timeout seen by any lane ends the role for the whole warp
  auto wait = [&](uint32_t b, uint32_t parity, unsigned site) {
    return __all_sync(0xffffffffu, mbar_wait(b, parity, wc, site));
  };
  // full / empty barriers of ring tile `it`
  auto wait_tile = [&](uint32_t it) {
    const bool ok = wait(bar(L::bKvFull + static_cast<int>(it % L::NS)), (it / L::NS) & 1u, kSiteMmaKv);
    tr.ev(p, kEvMmKv, it);
    return ok;
  };
  auto release_tile = [&](uint32_t it) { mma_commit(bar(L::bKvEmpty + static_cast<int>(it % L::NS)), leader); };

  const int num_tasks = task_count<VARLEN>(p);
  // short-task kernels with static assignment: the next task is decoded while
  // the current one runs, off the path from one task's last P V to the next
  // task's first Q K^T
  constexpr bool kPre = FD && !DYN;
  Task nxt{};
  if constexpr (kPre) {
    const int t0 = read_task<DQ, DV, DYN>(0, num_tasks, bar0, ring, wc, kSiteMmaTask);
    if (t0 >= 0) nxt = get_task<VARLEN, SPLIT, CAUSAL, FD, !DYN>(p, t0);
  }
  for (int kt = 0;; ++kt) {
    const int task = read_task<DQ, DV, DYN>(kt, num_tasks, bar0, ring, wc, kSiteMmaTask);
    if (task < 0) break;  // no task left, or an abort
    Task tk = kPre ? nxt : get_task<VARLEN, SPLIT, CAUSAL, FD, !DYN>(p, task);
    if (!check_task<CK>(p, tk, task, wc)) break;
    tr.ev(p, kEvMmTask, static_cast<uint32_t>(task));
    // decode task kt + 1 (called once the first Q K^T of task kt are issued)
    auto pre_next = [&]() {
      if constexpr (kPre) {
        const int t1 = read_task<DQ, DV, DYN>(kt + 1, num_tasks, bar0, ring, wc, kSiteMmaTask);
        if (t1 >= 0) nxt = get_task<VARLEN, SPLIT, CAUSAL, FD, !DYN>(p, t1);
      }
    };
    if (TS && tk.ksplit != 0) {
      // key-split tail task: both stages hold one Q tile and stream their own
      // key halves.  Ring order: K_0 of stage 0 and of stage 1, then per
      // block j and stage s: V_j, K_{j+1}.  Each tile is released right after
      // the MMA that reads it.
      uint32_t it = kv_it;
      kv_it += 2u * static_cast<uint32_t>(tk.n[0] + tk.n[1]);
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        if (!wait_tile(it)) goto out;
        if (!wait(bar(L::bQFull + s), q_phase[s], kSiteMmaQ)) goto out;
        q_phase[s] ^= 1u;
        cnt.inc(kCntMmQ + s);
        tc_fence_after();
        tr.ev(p, kEvMmQ, static_cast<uint32_t>(s));
        issue_qk<DQ, DV>(tmem + static_cast<uint32_t>(s * 128), q_addr(s), slot_addr(it), leader);
        mma_commit(bar(L::bSFull + s), leader);
        cnt.inc(kCntMmS + s);
        tr.ev(p, kEvMmQK, static_cast<uint32_t>(s << 16));
        if (tk.n[s] == 1) mma_commit(bar(L::bQEmpty + s), leader);
        release_tile(it++);
      }
      pre_next();
      for (int j = 0; j < tk.n[0]; ++j) {
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          if (j >= tk.n[s]) continue;
          if (!wait_tile(it)) goto out;
          if (!wait(bar(L::bPFull + s), p_phase[s], kSiteMmaP)) goto out;
          p_phase[s] ^= 1u;
          cnt.inc(kCntMmP + s);
          tc_fence_after();
          tr.ev(p, kEvMmP, static_cast<uint32_t>(s << 16 | j));
          issue_pv_half<DV>(tmem + 256u + static_cast<uint32_t>(s * 128), tmem + static_cast<uint32_t>(s * 128),
                            slot_addr(it), 0, j > 0, leader);
          issue_pv_half<DV>(tmem + 256u + static_cast<uint32_t>(s * 128), tmem + static_cast<uint32_t>(s * 128),
                            slot_addr(it), 1, true, leader);
          tr.ev(p, kEvMmPV, static_cast<uint32_t>(s << 16 | j));
          if (j + 1 == tk.n[s]) {
            mma_commit(bar(L::bODone + s), leader);
            cnt.inc(kCntMmODone + s);
          }
          release_tile(it++);
          if (j + 1 < tk.n[s]) {
            if (!wait_tile(it)) goto out;
            issue_qk<DQ, DV>(tmem + static_cast<uint32_t>(s * 128), q_addr(s), slot_addr(it), leader);
            mma_commit(bar(L::bSFull + s), leader);
            cnt.inc(kCntMmS + s);
            tr.ev(p, kEvMmQK, static_cast<uint32_t>(s << 16 | (j + 1)));
            if (j + 2 == tk.n[s]) mma_commit(bar(L::bQEmpty + s), leader);
            release_tile(it++);
          }
        }
      }
      continue;
    }
    const uint32_t base = kv_it;
    kv_it += 2u * static_cast<uint32_t>(tk.nmax);
    if (tk.nmax == 0) {
      pre_next();
      continue;
    }

    // prologue: S_s = Q_s K_0^T for both stages
    if (!wait_tile(base)) goto out;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      if (tk.n[s] == 0) continue;
      if (!wait(bar(L::bQFull + s), q_phase[s], kSiteMmaQ)) goto out;
      q_phase[s] ^= 1u;
      cnt.inc(kCntMmQ + s);
      tc_fence_after();
      tr.ev(p, kEvMmQ, static_cast<uint32_t>(s));
      issue_qk<DQ, DV>(tmem + static_cast<uint32_t>(s * 128), q_addr(s), slot_addr(base), leader);
      mma_commit(bar(L::bSFull + s), leader);
      cnt.inc(kCntMmS + s);
      tr.ev(p, kEvMmQK, static_cast<uint32_t>(s << 16));
      if (tk.n[s] == 1) mma_commit(bar(L::bQEmpty + s), leader);
    }
    release_tile(base);  // K_0, once both Q K^T have finished
    pre_next();

    for (int j = 0; j < tk.nmax; ++j) {
      const uint32_t v_it = base + 2u * static_cast<uint32_t>(j) + 1u;
      const uint32_t k_it = v_it + 1u;  // K_{j+1}
      if (!wait_tile(v_it)) goto out;
      bool k_ready = false;
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        if (j >= tk.n[s]) continue;
        if (!wait(bar(L::bPFull + s), p_phase[s], kSiteMmaP)) goto out;
        p_phase[s] ^= 1u;
        cnt.inc(kCntMmP + s);
        tc_fence_after();
        tr.ev(p, kEvMmP, static_cast<uint32_t>(s << 16 | j));
        issue_pv_half<DV>(tmem + 256u + static_cast<uint32_t>(s * 128), tmem + static_cast<uint32_t>(s * 128),
                          slot_addr(v_it), 0, j > 0, leader);
        issue_pv_half<DV>(tmem + 256u + static_cast<uint32_t>(s * 128), tmem + static_cast<uint32_t>(s * 128),
                          slot_addr(v_it), 1, true, leader);
        tr.ev(p, kEvMmPV, static_cast<uint32_t>(s << 16 | j));
        if (j + 1 == tk.n[s]) {
          mma_commit(bar(L::bODone + s), leader);
          cnt.inc(kCntMmODone + s);
        }
        // with a shallow ring (d_qk = 192: two slots) V_j's slot is released
        // by the last P V that reads it, so that V_{j+1} can be loaded while
        // the next Q K^T runs; with a deeper ring the release waits for the
        // block's end (measured: +13 % at d_qk = 192, -1 % at 128)
        if constexpr (kEarlyV) {
          if (s == 1 || j >= tk.n[1]) release_tile(v_it);
        }
        if (j + 1 < tk.n[s]) {
          if (!k_ready) {
            if (!wait_tile(k_it)) goto out;
            k_ready = true;
          }
          issue_qk<DQ, DV>(tmem + static_cast<uint32_t>(s * 128), q_addr(s), slot_addr(k_it), leader);
          mma_commit(bar(L::bSFull + s), leader);
          cnt.inc(kCntMmS + s);
          tr.ev(p, kEvMmQK, static_cast<uint32_t>(s << 16 | (j + 1)));
          if (j + 2 == tk.n[s]) mma_commit(bar(L::bQEmpty + s), leader);
        }
      }
      // V_j (deep ring), and K_{j+1} once its Q K^T have finished
      if constexpr (!kEarlyV) release_tile(v_it);
      if (j + 1 < tk.nmax) release_tile(k_it);
    }
  }
out:
  // every MMA issued by the leader lane has completed once the drain barrier fires
  mma_commit(bar(L::bDrain), leader);
  mbar_drain_wait(bar(L::bDrain), 0u, wc, kSiteMmaDrain);
  tr.finish(p);
  if (!*wc.abort_flag) {
    cnt.add(kCntMmKv, kv_it);
    cnt.store(dbg_area, kCntMmKv, kCntMmODone + 2, leader != 0);
  }
}

// ---------------------------------------------------------------------------
// TMA loads (warp 13, one thread)
// ---------------------------------------------------------------------------
template <int DQ, int DV, bool CAUSAL, bool VARLEN, bool DYN, bool SPLIT, bool FD, int VAR>
__device__ __forceinline__ void load_role(const Params& p, const uint32_t sbase, volatile int* ring,
                                          uint32_t* dbg_area, const WaitCtx& wc) {
  using L = Layout<DQ, DV>;
  constexpr bool CK = (VAR & kVarCheck) != 0;
  const Problem& pr = p.prob;
  Tracer<(VAR & kVarTrace) != 0, 4> tr;
  tr.init(p, true);
  constexpr bool TS = !CAUSAL && !VARLEN && !DYN && !SPLIT;  // key-split tail tasks possible
  const uint32_t bar0 = sbase + L::oBar;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t q_uses[2] = {0u, 0u};
  uint32_t kv_it = 0;  // K/V tiles issued

  tma_prefetch_desc(&p.tm_q);
  tma_prefetch_desc(&p.tm_k);
  tma_prefetch_desc(&p.tm_v);

  const int num_tasks = task_count<VARLEN>(p);
  for (int kt = 0;; ++kt) {
    const int task = post_task<DQ, DV, DYN>(p, kt, num_tasks, bar0, ring, wc);
    if (task < 0) break;  // no task left, or an abort
    Task tk = get_task<VARLEN, SPLIT, CAUSAL, FD, !DYN>(p, task);
    if (!check_task<CK>(p, tk, task, wc)) break;
    tr.ev(p, kEvLdTask, static_cast<uint32_t>(task));
    if (tk.nmax == 0) continue;
    // Q tile of stage s (none when the stage has no block)
    auto load_q = [&](int s) -> bool {
      if (tk.n[s] == 0) return true;
      if (q_uses[s] > 0 && !mbar_wait(bar(L::bQEmpty + s), (q_uses[s] - 1u) & 1u, wc, kSiteLoadQ)) return false;
      if constexpr (CK) {  // the Q tile starts inside q
        const int row = tk.q_row0 + tk.pos0[s];
        if (!dbg_check(row >= 0 && row < pr.Sq && tk.g >= 0 && tk.g < pr.groups && tk.bc >= 0 && tk.bc < pr.B, wc,
                       kSiteCheckQCoord))
          return false;
      }
      const uint32_t qb = bar(L::bQFull + s);
      mbar_arrive_expect_tx(qb, L::NQC * kChunkBytes);
      const uint32_t dst = sbase + L::oQ + static_cast<uint32_t>(s * L::kQBytes);
      for (int c = 0; c < L::NQC; ++c)
        tma_load_5d(dst + c * kChunkBytes, &p.tm_q, qb, c * 64, 0, tk.g, tk.q_row0 + tk.pos0[s], tk.bc);
      ++q_uses[s];
      tr.ev(p, kEvLdQ, static_cast<uint32_t>(s));
      return true;
    };
    // K_j (which = 0) or V_j (1) into the next ring slot
    auto load_kv = [&](int which, int j) -> bool {
      const uint32_t slot = kv_it % L::NS;
      tr.ev(p, kEvLdKvWait, kv_it);
      if (kv_it >= static_cast<uint32_t>(L::NS) &&
          !mbar_wait(bar(L::bKvEmpty + static_cast<int>(slot)), ((kv_it / L::NS) - 1u) & 1u, wc, kSiteLoadKv))
        return false;
      if constexpr (CK) {  // the K/V tile starts inside k / v
        const int row = tk.k_row0 + j * kBN;
        if (!dbg_check(row >= 0 && row < pr.Sk && tk.kvh >= 0 && tk.kvh < pr.Hkv && tk.bc >= 0 && tk.bc < pr.B, wc,
                       kSiteCheckKvCoord))
          return false;
      }
      const uint32_t fb = bar(L::bKvFull + static_cast<int>(slot));
      const uint32_t dst = sbase + L::oRing + slot * L::kSlotBytes;
      const int nch = which == 0 ? L::NQC : L::NVC;
      mbar_arrive_expect_tx(fb, static_cast<uint32_t>(nch * kChunkBytes));
      for (int c = 0; c < nch; ++c)
        tma_load_4d(dst + c * kChunkBytes, which == 0 ? static_cast<const void*>(&p.tm_k) : &p.tm_v, fb, c * 64,
                    tk.kvh, tk.k_row0 + j * kBN, tk.bc);
      tr.ev(p, kEvLdKv, kv_it);
      ++kv_it;
      return true;
    };
    if (!load_q(0) || !load_q(1)) goto out;
    if constexpr (TS) {
      if (tk.ksplit != 0) {  // key-split tail task: the order the MMA warp reads
        // the next ring tile: K (which = 0) or V (1) of the block at key row `row`
        auto issue_tile = [&](int which, int row) -> bool {
          const uint32_t slot = kv_it % L::NS;
          tr.ev(p, kEvLdKvWait, kv_it);
          if (kv_it >= static_cast<uint32_t>(L::NS) &&
              !mbar_wait(bar(L::bKvEmpty + static_cast<int>(slot)), ((kv_it / L::NS) - 1u) & 1u, wc, kSiteLoadKv))
            return false;
          if constexpr (CK) {  // the K/V tile starts inside k / v
            if (!dbg_check(row >= 0 && row < pr.Sk && tk.kvh >= 0 && tk.kvh < pr.Hkv && tk.bc >= 0 && tk.bc < pr.B,
                           wc, kSiteCheckKvCoord))
              return false;
          }
          const uint32_t fb = bar(L::bKvFull + static_cast<int>(slot));
          const uint32_t dst = sbase + L::oRing + slot * L::kSlotBytes;
          const int nch = which == 0 ? L::NQC : L::NVC;
          mbar_arrive_expect_tx(fb, static_cast<uint32_t>(nch * kChunkBytes));
          for (int c = 0; c < nch; ++c)
            tma_load_4d(dst + c * kChunkBytes, which == 0 ? static_cast<const void*>(&p.tm_k) : &p.tm_v, fb,
                        c * 64, tk.kvh, row, tk.bc);
          tr.ev(p, kEvLdKv, kv_it);
          ++kv_it;
          return true;
        };
        const int row1 = tk.k_row0 + tk.ksplit * kBN;  // stage 1's first key
        if (!issue_tile(0, tk.k_row0) || !issue_tile(0, row1)) goto out;
        for (int j = 0; j < tk.n[0]; ++j) {
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            if (j >= tk.n[s]) continue;
            const int row = (s ? row1 : tk.k_row0) + j * kBN;
            if (!issue_tile(1, row)) goto out;
            if (j + 1 < tk.n[s] && !issue_tile(0, row + kBN)) goto out;
          }
        }
        continue;
      }
    }
    for (int j = 0; j < tk.nmax; ++j) {
#pragma unroll
      for (int which = 0; which < 2; ++which) {  // K_j then V_j
        if (!load_kv(which, j)) goto out;
      }
    }
  }
out:
  // drain: the last copy issued into every buffer has landed
#pragma unroll
  for (int s = 0; s < 2; ++s)
    if (q_uses[s] > 0) mbar_drain_wait(bar(L::bQFull + s), (q_uses[s] - 1u) & 1u, wc, kSiteLoadDrain);
  for (uint32_t i = 0; i < static_cast<uint32_t>(L::NS) && i < kv_it; ++i) {
    const uint32_t uses = (kv_it - i + L::NS - 1) / L::NS;  // copies issued into slot i
    mbar_drain_wait(bar(L::bKvFull + static_cast<int>(i)), (uses - 1u) & 1u, wc, kSiteLoadDrain);
  }
  tr.finish(p);
  if constexpr (CK) {
    if (!*wc.abort_flag) {
      dbg_area[kCntLdKv] = kv_it;
      dbg_area[kCntLdQ] = q_uses[0];
      dbg_area[kCntLdQ + 1] = q_uses[1];
    }
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int DQ, int DV, bool CAUSAL, int MODE, int VAR>
__global__ void __launch_bounds__(kThreads, 1) fa_fwd_kernel(const __grid_constant__ Params p) {
  using L = Layout<DQ, DV>;
  static_assert(VAR == 0 || MODE == kModeFixed || MODE == kModeDirect, "build variants: fixed-length modes only");
  static_assert(256 + 128 + DV <= static_cast<int>(kTmemCols), "S0, S1, O0 and O1 fit in TMEM");
  constexpr bool CK = (VAR & kVarCheck) != 0;
  constexpr bool EMU = MODE == kModeEmu;
  constexpr bool VARLEN = MODE == kModeVarlen;
  constexpr bool DYN = MODE == kModeVarlen || MODE == kModeDyn;
  constexpr bool SPLIT = MODE == kModeSplit;
  constexpr bool DIRECT = MODE == kModeDirect;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::oMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::oMisc + 4);
  float* mbox = reinterpret_cast<float*>(smem + L::oMbox);
  volatile int* ring = reinterpret_cast<volatile int*>(smem + L::oTaskRing);
  uint32_t* dbg_area = reinterpret_cast<uint32_t*>(smem + L::oDbgCount);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    if constexpr (CK) {
      for (int i = 0; i < kNumCounts; ++i) dbg_area[i] = 0u;
    }
    const uint32_t b = sbase + L::oBar;
    for (int s = 0; s < 2; ++s) {
      mbar_init(b + 8 * (L::bQFull + s), 1);
      mbar_init(b + 8 * (L::bQEmpty + s), 1);
      mbar_init(b + 8 * (L::bSFull + s), 1);
      mbar_init(b + 8 * (L::bPFull + s), 256);
      mbar_init(b + 8 * (L::bODone + s), 1);
      mbar_init(b + 8 * (L::bCorrFull + s), 128);
      mbar_init(b + 8 * (L::bFinFull + 2 * s), 128);
      mbar_init(b + 8 * (L::bFinFull + 2 * s + 1), 128);
      mbar_init(b + 8 * (L::bStagger + s), 128);
    }
    for (int i = 0; i < L::NS; ++i) {
      mbar_init(b + 8 * (L::bKvFull + i), 1);
      mbar_init(b + 8 * (L::bKvEmpty + i), 1);
    }
    mbar_init(b + 8 * L::bEpiFull, 128);
    mbar_init(b + 8 * L::bStageFree, 1);
    mbar_init(b + 8 * L::bDrain, 1);
    mbar_init(b + 8 * L::bSink, 256);
    for (int r = 0; r < kTaskRing; ++r) {
      mbar_init(b + 8 * (L::bTaskFull + r), 1);
      mbar_init(b + 8 * (L::bTaskEmpty + r), kTaskReaders);
    }
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 12) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};
  if constexpr (CK) {
    if (threadIdx.x == 0) {
      // the aligned layout ends inside the launch's dynamic shared memory
      uint32_t dyn_bytes;
      asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn_bytes));
      dbg_check(static_cast<uint32_t>(smem - smem_raw) + static_cast<uint32_t>(L::kBytes) <= dyn_bytes, wc,
                kSiteCheckSmem);
      // all 512 columns were allocated, so the base is lane 0, column 0
      dbg_check(tmem == 0u, wc, kSiteCheckTmem);
    }
    __syncthreads();
  }

  // register budget: 128 x (176 + 176 + 104 + 56) = 65536
  if (warp < 8) {
    setmaxnreg_inc<176>();
    softmax_role<DQ, DV, CAUSAL, EMU, VARLEN, DYN, SPLIT, DIRECT, VAR>(p, warp >> 2, tmem, sbase, mbox, ring,
                                                                      dbg_area, wc);
  } else if (warp < 12) {
    setmaxnreg_dec<104>();
    correction_role<DQ, DV, CAUSAL, VARLEN, DYN, SPLIT, DIRECT, EMU || (VAR & kVarCheck) != 0, VAR>(p, tmem, sbase, smem, mbox, ring,
                                                                           dbg_area, wc);
  } else {
    setmaxnreg_dec<56>();
    if (warp == 12) {
      mma_role<DQ, DV, CAUSAL, VARLEN, DYN, SPLIT, DIRECT, VAR>(p, tmem, sbase, ring, dbg_area, wc);
      __syncwarp();
    } else if (warp == 13) {
      if (lane == 0) load_role<DQ, DV, CAUSAL, VARLEN, DYN, SPLIT, DIRECT, VAR>(p, sbase, ring, dbg_area, wc);
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (CK) {
    // every hand-off was produced as often as it was consumed
    if (threadIdx.x == 0 && !*abort_flag) {
      const uint32_t* c = dbg_area;
      const bool same[] = {
          c[kCntLdKv] == c[kCntMmKv],           c[kCntLdQ] == c[kCntMmQ],
          c[kCntLdQ + 1] == c[kCntMmQ + 1],     c[kCntMmS] == c[kCntSmS],
          c[kCntMmS + 1] == c[kCntSmS + 1],     c[kCntSmS] == c[kCntCoCorr],
          c[kCntSmS + 1] == c[kCntCoCorr + 1],  c[kCntSmP] == c[kCntMmP],
          c[kCntSmP + 1] == c[kCntMmP + 1],     c[kCntCoP] == c[kCntMmP],
          c[kCntCoP + 1] == c[kCntMmP + 1],     c[kCntMmODone] == c[kCntCoODone],
          c[kCntMmODone + 1] == c[kCntCoODone + 1]};
      for (int i = 0; i < static_cast<int>(sizeof(same) / sizeof(same[0])); ++i)
        if (!dbg_check(same[i], wc, kSiteCheckCounts + static_cast<unsigned>(i))) break;
    }
  }
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace fa
