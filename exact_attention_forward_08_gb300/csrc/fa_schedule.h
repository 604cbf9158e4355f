// Tile decomposition and task order of the attention forward kernel.
//
// Shared by the host (plan, launch) and the device (each persistent CTA walks
// task indices blockIdx.x, blockIdx.x + gridDim.x, ...).  Plain integer
// arithmetic, compiled for both sides so that the host tests check exactly
// what the kernel runs.
//
// Decomposition ("Flash Attention 4 on Blackwell", sections "Causal attention
// and GQA" and "Scheduling"):
//  * A Q tile has BM = 128 rows.  With GQA/MQA the 128 rows pack `pack` query
//    heads that share one KV head: row r is sequence position pos0 + r / pack
//    of query head g * pack + r % pack, so K/V are never replicated.  pack is
//    the GQA ratio when it divides 128, else 1 (one query head per tile, which
//    keeps every integer ratio supported).
//  * A task is (batch b, head group g, m_block): two consecutive Q tiles
//    (stage 0 and stage 1) that stream the same K/V blocks.
//  * n_blocks(stage) is the number of 128-key blocks the tile visits: all of
//    them without a mask; under the bottom-right causal mask only blocks that
//    hold a key j <= pos_last + Sk - Sq (future blocks are skipped).
//  * Task order: linear for the non-causal case (uniform cost).  For the
//    causal case longest-processing-time first: the heavier half of the
//    m_blocks (m >= M - ceil(M/2)) in decreasing order inside sections of
//    `section_units` (b, g) units whose K/V fill a section budget (about
//    8 MiB, well inside L2: causal_section_budget), then the
//    lighter half level by level (m decreasing, all units per level).  Light
//    tasks read only the first half of a unit's K/V, and ending the list with
//    the cheapest tasks keeps the last CTAs from finishing late (a static
//    round-robin over "heaviest first per section" alone left the busiest CTA
//    with 11-29 % more work than the average; this order halves that, and a
//    dynamic assignment over it comes within about 1 %).
//  * Balanced last wave (non-causal fixed-length problems): with P tasks on
//    G persistent CTAs taken round-robin, the last r = P mod G tasks form a
//    partial wave that keeps G - r CTAs idle while the others run a whole
//    task.  When 2r <= G, each tile of those r tasks becomes a task of its
//    own whose two stages hold the same Q tile and the two halves of the key
//    blocks; the epilogue merges the two halves' (row max, row sum, O) with
//    the exact rescaling of the online softmax ("Infra: Flash Attention",
//    "Prefill and decode": independently computed key segments merge
//    exactly).  The last wave then takes about half a task instead of one.
//  * Paired causal order (static assignment): m_blocks m and M-1-m of a unit
//    see (2m + 1.5) and (2M - 2m - 0.5) key blocks on average, a constant
//    sum.  With M even, the list is laid out for G CTAs in blocks of 2G
//    entries: G light tasks followed by their G heavy complements (pair i:
//    the i-th task of the heavier half in the L2-section order above and its
//    complement), so that CTA c runs the light task of pair bG + c and then
//    its heavy complement, which re-reads the K/V prefix the light task just
//    brought into L2 before streaming the rest; every CTA then gets the same
//    work per two waves.  The r = P mod G pairs
//    left over (P = units * M / 2) go last.  When 2r <= G each pair's two
//    tasks go to two CTAs.  Otherwise the left-over pairs are taken from the
//    heaviness levels whose heavy task costs about r / G of a pair: their
//    heavy tasks run on CTAs 0 .. r-1 and their light complements are dealt
//    round-robin over the G - r other CTAs (about r / (G - r) each), so the
//    last wave costs about r / G of a pair instead of a whole one; the list
//    then holds empty entries where a CTA has nothing left.  The levels are
//    chosen on the host with a cost model (key blocks of the two tiles / 2
//    plus a fixed start-up per task); when no choice beats keeping each pair
//    on one CTA, that is what runs.  The model put the busiest CTA 6-13 %
//    above the average with the plain order on the causal benchmark problems,
//    3.9 % with pairs alone and 0.5-1.8 % with the packed last wave.
//  * Split-KV (decode and other short-Q problems, where (b, g, m_block) tasks
//    are too few to fill the GPU): each task also takes one of `splits`
//    consecutive key ranges of split_blocks blocks ("Infra: Flash Attention",
//    "Prefill and decode": the state merge does not fix the scan order, so
//    the keys can be cut into segments computed apart and merged after); the
//    partial results are combined by a separate merge kernel.
//  * Variable-length batches (sequences packed back to back, offsets in
//    cu_seqlens): a planning kernel sorts the sequences by the cost of their
//    heaviest tile, longest first ("FlashAttention-4 wiki", "Core methods",
//    LPT scheduling: varlen batches are ordered by a preprocessing kernel),
//    and lists every sequence's tasks in the order above, one sequence after
//    the other.  The persistent CTAs then walk that list.
#pragma once
#include <cstdint>

#ifdef __CUDACC__
#define FA_HD __host__ __device__ __forceinline__
#else
#define FA_HD inline
#endif

namespace fa {

constexpr int kBM = 128;  // rows of a Q tile (TMEM lanes)
constexpr int kBN = 128;  // keys of a K/V block

// Division by a divisor fixed when the problem is planned, as a multiply and
// a shift (the round-up method of Granlund and Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994): for 0 <= n < 2^31 and
// 1 <= d <= 2^31, with L = ceil(log2 d) and m = ceil(2^(31+L) / d) (which is
// below 2^32), floor(n / d) = floor(n * m / 2^(31+L)), because the error
// n * (m d - 2^(31+L)) / (d 2^(31+L)) stays below 1/d.  A run-time integer
// division compiles to a reciprocal on the SFU, the pipe the softmax keeps
// busy with exponentials, so the kernel's task decoding uses these instead.
struct FastDiv {
  uint32_t m;
  uint32_t shift;
};

FA_HD FastDiv make_fastdiv(int d) {
  if (d < 1) d = 1;
  uint32_t L = 0;
  while ((uint64_t(1) << L) < static_cast<uint64_t>(d)) ++L;
  const uint64_t num = uint64_t(1) << (31 + L);
  FastDiv f;
  f.m = static_cast<uint32_t>((num + static_cast<uint64_t>(d) - 1) / static_cast<uint64_t>(d));
  f.shift = 31 + L;
  return f;
}

// floor(n / d) for 0 <= n < 2^31
FA_HD int fdiv(int n, FastDiv f) {
  return static_cast<int>((static_cast<uint64_t>(static_cast<uint32_t>(n)) * f.m) >> f.shift);
}

struct Problem {
  int B, Hq, Hkv, Sq, Sk;
  int causal;
  int pack;           // query heads per Q tile
  int groups;         // Hq / pack
  int pos_per_tile;   // kBM / pack
  int tiles;          // Q tiles per (b, g): ceil(Sq / pos_per_tile)
  int mblocks;        // tasks per (b, g): ceil(tiles / 2)
  int kv_blocks;      // ceil(Sk / kBN)
  int ratio;          // Hq / Hkv
  int section_units;  // causal task order: (b, g) units per L2 section
  int heavy_levels;   // causal task order: m_blocks M-1 .. M-heavy_levels go by sections
  int splits;         // split-KV: key ranges per (b, g, m_block) (1 = no split)
  int split_blocks;   // split-KV: K/V blocks per range
  int64_t num_tasks;  // B * groups * mblocks * splits (+ the key-split tail tasks)
  int64_t tail_first; // first key-split tail task (= num_tasks when there are none)
  // paired causal order (set_pairing): 0 = the plain longest-first order
  int pair_grid;       // CTAs the paired list is laid out for
  int pair_body;       // entries of the whole blocks (2 * G * (P / G))
  int pair_r;          // pairs left over (P mod G)
  int pair_split_tail; // 1: each left-over pair's two tasks go to two CTAs
  int pair_pack;       // 1: left-over heavy tasks on r CTAs, their complements on the others
  int pair_q0, pair_nt;// pair_nt > 0: heaviness levels q0 .. q0+nt-1 go last (the left-over pairs)
  // the divisors of the task decoding (set_divisors)
  FastDiv fd_mblocks, fd_splits, fd_groups, fd_ratio, fd_pack;
  FastDiv fd_units;    // B * groups
  FastDiv fd_section;  // section_units * heavy_levels
  FastDiv fd_su;       // section_units
  FastDiv fd_last;     // units of the last causal section
  FastDiv fd_pair2g;   // 2 * pair_grid
  FastDiv fd_grid;     // pair_grid
  FastDiv fd_section_main;  // section_units * (heavy_levels - pair_nt)
};

// Fill the FastDiv fields from the integer fields; call after any change.
FA_HD void set_divisors(Problem& p) {
  const int units = p.B * p.groups;
  p.fd_mblocks = make_fastdiv(p.mblocks);
  p.fd_splits = make_fastdiv(p.splits);
  p.fd_groups = make_fastdiv(p.groups);
  p.fd_ratio = make_fastdiv(p.ratio);
  p.fd_pack = make_fastdiv(p.pack);
  p.fd_units = make_fastdiv(units);
  p.fd_section = make_fastdiv(p.section_units * p.heavy_levels);
  p.fd_su = make_fastdiv(p.section_units);
  const int su = p.section_units > 0 ? p.section_units : 1;
  const int last_first = units > 0 ? ((units - 1) / su) * su : 0;
  p.fd_last = make_fastdiv(units - last_first);
  p.fd_pair2g = make_fastdiv(2 * (p.pair_grid > 0 ? p.pair_grid : 1));
  p.fd_grid = make_fastdiv(p.pair_grid > 0 ? p.pair_grid : 1);
  p.fd_section_main = make_fastdiv(p.section_units * (p.heavy_levels - p.pair_nt));
}

struct Task {
  int b, g, mb;
  int kvh;       // K/V head read by this task
  int pos0[2];   // first sequence position of each stage's tile
  int n[2];      // K/V blocks each stage visits (0: nothing to do)
  int nmax;      // max(n[0], n[1])
  int sq;        // query count of this task's sequence
  // keys of the task, counted from its first key: those >= kend are never
  // visible; under the causal mask position pos sees key r iff r <= pos + kshift
  // (a whole sequence: kend = sk, kshift = sk - sq; split-KV range starting at
  // key k0: kend = its length, kshift = sk - sq - k0)
  int kend, kshift;
  int q_row0;    // row of position 0 in the Q/O view (varlen: cu_seqlens_q[b]; else 0)
  int k_row0;    // row of the task's first key in the K/V view
  int bc;        // batch coordinate in the TMA views (varlen: 0; else b)
  int split;     // split-KV range index (0 otherwise)
  int ksplit;    // key-split tail task: both stages hold the tile at pos0[0]; stage 0
                 // visits key blocks [0, ksplit), stage 1 [ksplit, ksplit + n[1]).
                 // 0 for every other task.
};

// One task of a variable-length batch as the planning kernel writes it
// (32 bytes, read with two 16-byte loads).
struct alignas(16) VarlenTask {
  int b, g, mb, reserved;
  int q_row0, sq, k_row0, sk;
};

FA_HD int ceil_div(int a, int b) { return (a + b - 1) / b; }

FA_HD int choose_pack(int Hq, int Hkv) {
  const int ratio = Hq / Hkv;
  return (ratio >= 1 && kBM % ratio == 0) ? ratio : 1;
}

// Fill the derived fields.  `pack_override` > 0 forces a pack (must divide
// both 128 and the ratio); l2_budget_bytes sizes the causal sections.  The
// FastDiv fields are left for make_problem (the varlen planner builds a
// problem per task record and decodes with plain division).
FA_HD Problem make_problem_core(int B, int Hq, int Hkv, int Sq, int Sk, int d_qk, int d_v, int causal,
                                int64_t l2_budget_bytes, int pack_override) {
  Problem p{};  // FastDiv fields zero until set_divisors
  p.B = B, p.Hq = Hq, p.Hkv = Hkv, p.Sq = Sq, p.Sk = Sk, p.causal = causal;
  p.ratio = Hq / Hkv;
  p.pack = pack_override > 0 ? pack_override : choose_pack(Hq, Hkv);
  p.groups = Hq / p.pack;
  p.pos_per_tile = kBM / p.pack;
  p.tiles = ceil_div(Sq, p.pos_per_tile);
  p.mblocks = ceil_div(p.tiles, 2);
  p.kv_blocks = ceil_div(Sk, kBN);
  p.num_tasks = static_cast<int64_t>(B) * p.groups * p.mblocks;
  p.tail_first = p.num_tasks;
  // K/V bytes one (b, g) unit streams; units that share a KV head (pack = 1
  // with GQA) share those bytes in L2, which only makes the estimate safe.
  const int64_t kv_bytes = static_cast<int64_t>(Sk) * (d_qk + d_v) * 2;
  int64_t su = kv_bytes > 0 ? l2_budget_bytes / kv_bytes : 1;
  const int64_t units = static_cast<int64_t>(B) * p.groups;
  if (su < 1) su = 1;
  if (su > units) su = units > 0 ? units : 1;
  p.section_units = static_cast<int>(su);
  p.heavy_levels = (p.mblocks + 1) / 2;
  p.splits = 1;
  p.split_blocks = p.kv_blocks;
  return p;
}

// K/V bytes per section of the fixed-length causal order: about 8 MiB (at
// most half the L2).  Measured on GB300 (L2 126 MiB) against half the L2:
// causal 2k and 8k +2 %, 4k +1.5 %, 1k +0.8 %, 16k +0.4 %, 32k -0.4 %, GQA /
// MQA / (192, 128) within +-0.3 % (2 or 4 MiB: causal 8k -1 %, 4k -3 % at
// 2 MiB).  Few units per section keep the CTAs that run at one time on the
// K/V of few units, which they then read out of L2 together.
constexpr int64_t kCausalSectionBytes = int64_t(8) << 20;
FA_HD int64_t causal_section_budget(int64_t l2_bytes) {
  const int64_t half = l2_bytes / 2;
  return half < kCausalSectionBytes ? half : kCausalSectionBytes;
}

FA_HD Problem make_problem(int B, int Hq, int Hkv, int Sq, int Sk, int d_qk, int d_v, int causal,
                           int64_t l2_budget_bytes, int pack_override) {
  Problem p = make_problem_core(B, Hq, Hkv, Sq, Sk, d_qk, d_v, causal, l2_budget_bytes, pack_override);
  set_divisors(p);
  return p;
}

// Split the keys of every (b, g, m_block) into about `splits` ranges of whole
// blocks (no empty range: the count is recomputed from the range length).
FA_HD void set_splits(Problem& p, int splits) {
  if (splits < 1 || p.kv_blocks == 0) splits = 1;
  if (splits > p.kv_blocks && p.kv_blocks > 0) splits = p.kv_blocks;
  p.split_blocks = p.kv_blocks > 0 ? ceil_div(p.kv_blocks, splits) : 0;
  p.splits = p.split_blocks > 0 ? ceil_div(p.kv_blocks, p.split_blocks) : 1;
  p.num_tasks = static_cast<int64_t>(p.B) * p.groups * p.mblocks * p.splits;
  p.tail_first = p.num_tasks;
  set_divisors(p);
}

// Balanced last wave: a non-causal problem of P (b, g, m_block) tasks run by
// `grid` CTAs round-robin (task t on CTA t mod grid) ends with a partial wave
// of r = P mod grid tasks (r = P when P < grid).  When 0 < 2r <= grid, the
// last r tasks are replaced by 2r key-split tasks, one per tile: task
// tail_first + 2i + u runs tile u of pair task tail_first + i with the keys
// halved over the two stages.  Needs at least kTailSplitMinBlocks K/V blocks
// (both halves non-empty, and enough keys to pay for the merge).
constexpr int kTailSplitMinBlocks = 4;

FA_HD int tail_split_pairs(const Problem& p, int64_t grid) {
  if (p.causal || p.splits != 1 || p.kv_blocks < kTailSplitMinBlocks || grid < 2) return 0;
  const int64_t P = p.num_tasks;
  const int64_t r = P >= grid ? P % grid : P;
  return (r > 0 && 2 * r <= grid) ? static_cast<int>(r) : 0;
}

FA_HD void set_tail_split(Problem& p, int64_t grid) {
  const int r = tail_split_pairs(p, grid);
  if (r == 0) return;
  p.tail_first = p.num_tasks - r;
  p.num_tasks += r;
}


// K/V blocks a Q tile starting at pos0 visits (sq queries, ppt positions per
// tile; kend / kshift as in Task).
FA_HD int tile_blocks_len(int sq, int kend, int kshift, int causal, int ppt, int pos0) {
  if (pos0 >= sq || kend <= 0) return 0;
  const int kvb = ceil_div(kend, kBN);
  if (!causal) return kvb;
  int last = pos0 + ppt;
  if (last > sq) last = sq;
  const int64_t max_key = static_cast<int64_t>(last - 1) + kshift;
  if (max_key < 0) return 0;
  const int64_t n = max_key / kBN + 1;
  return n < kvb ? static_cast<int>(n) : kvb;
}

// Paired causal order for `grid` CTAs taken round-robin (see the header
// comment): needs an even m_block count and a list that stays below 2^31.
// Modelled cost of m_block m: key blocks of its two tiles / 2 + a start-up.
constexpr double kPairTaskStartup = 2.5;

FA_HD double pair_task_cost(const Problem& p, int m) {
  const int kshift = p.Sk - p.Sq;
  const int a = tile_blocks_len(p.Sq, p.Sk, kshift, 1, p.pos_per_tile, (2 * m) * p.pos_per_tile);
  const int b = tile_blocks_len(p.Sq, p.Sk, kshift, 1, p.pos_per_tile, (2 * m + 1) * p.pos_per_tile);
  return 0.5 * (a + b) + kPairTaskStartup;
}

// Modelled last wave when the r left-over pairs come from heaviness levels
// q0 .. q0+nt-1 (the last r pairs of those levels, level-major over units):
// heavy tasks one per CTA, light complements round-robin over G - r CTAs.
FA_HD double packed_tail_cost(const Problem& p, int G, int r, int q0, int nt) {
  const int M = p.mblocks, units = p.B * p.groups;
  double worst = 0.0;
  for (int j = 0; j < r; ++j) {  // heavy tasks
    const int q = q0 + (nt * units - r + j) / units;
    const double h = pair_task_cost(p, M - 1 - q);
    if (h > worst) worst = h;
  }
  const int free = G - r;
  for (int c = 0; c < free; ++c) {  // light loads
    double load = 0.0;
    for (int j = c; j < r; j += free) load += pair_task_cost(p, q0 + (nt * units - r + j) / units);
    if (load > worst) worst = load;
  }
  return worst;
}

FA_HD void set_pairing(Problem& p, int64_t grid) {
  if (!p.causal || p.splits != 1 || p.mblocks < 2 || (p.mblocks & 1) || grid < 2 || p.pair_grid != 0) return;
  const int64_t P = static_cast<int64_t>(p.B) * p.groups * (p.mblocks / 2);
  const int64_t full = P / grid, r = P % grid;
  const bool split_tail = 2 * r <= grid;
  int pack = 0, q0 = 0, nt = 0;
  int64_t tail = r == 0 ? 0 : (split_tail ? 2 * r : grid + r);
  if (!split_tail && grid <= (int64_t(1) << 20)) {  // try packing the light complements
    const int units = p.B * p.groups, Mh = p.mblocks / 2, G = static_cast<int>(grid), R = static_cast<int>(r);
    const int need = (R + units - 1) / units;  // heaviness levels that hold r pairs
    const int M = p.mblocks;
    double best = pair_task_cost(p, M - 1) + pair_task_cost(p, 0);  // a whole pair on one CTA
    if (need <= Mh) {
      for (int c = 0; c + need <= Mh; ++c) {
        const double cost = packed_tail_cost(p, G, R, c, need);
        if (cost < 0.999 * best) best = cost, pack = 1, q0 = c, nt = need;
      }
    }
    if (pack) tail = ((r + (grid - r) - 1) / (grid - r)) * grid;
  }
  const int64_t n = 2 * full * grid + tail;
  if (n >= (int64_t(1) << 31)) return;
  p.pair_grid = static_cast<int>(grid);
  p.pair_body = static_cast<int>(2 * full * grid);
  p.pair_r = static_cast<int>(r);
  p.pair_split_tail = split_tail ? 1 : 0;
  p.pair_pack = pack;
  p.pair_q0 = q0;
  p.pair_nt = nt;
  p.num_tasks = n;
  p.tail_first = n;
  set_divisors(p);
}

// The balanced static order for `grid` CTAs: the key-split last wave without
// the mask, the paired order with it.
FA_HD void set_balance(Problem& p, int64_t grid) {
  if (p.causal) set_pairing(p, grid);
  else set_tail_split(p, grid);
}

// Task t (0 <= t < num_tasks < 2^31; the host refuses larger problems).
// CAUSAL is the mask kind when the caller knows it at compile time (0 or 1),
// or -1 to read p.causal.  FAST divides with the FastDiv fields; the result is
// the same either way (FastDiv is exact in this range).  TAIL decodes the
// key-split last wave (no mask), PAIR the paired order (causal mask); callers
// that never see them, such as the dynamically scheduled kernels, leave that
// code out.
template <int CAUSAL, bool FAST, bool TAIL = true, bool PAIR = true>
FA_HD Task decode_task_k(const Problem& p, int t) {
  const bool causal = CAUSAL < 0 ? p.causal != 0 : CAUSAL != 0;
  Task k;
  const int M = p.mblocks;
  int unit, mb;
  int tail_tile = -1;  // key-split tail task: the tile (0 or 1) of its pair task
  if (!causal) {
    if (TAIL && t >= p.tail_first) {
      const int u = t - static_cast<int>(p.tail_first);
      tail_tile = u & 1;
      t = static_cast<int>(p.tail_first) + (u >> 1);
    }
    unit = FAST ? fdiv(t, p.fd_mblocks) : t / M;
    mb = t - unit * M;
  } else {
    bool light = false;  // paired order: the light complement of pair t
    if (PAIR && p.pair_grid > 0) {
      const int G = p.pair_grid;
      if (t < p.pair_body) {  // blocks of G light complements and their G heavy tasks
        const int blk = FAST ? fdiv(t, p.fd_pair2g) : t / (2 * G);
        const int w = t - blk * 2 * G;
        light = w < G;
        t = blk * G + (light ? w : w - G);
      } else {  // the pairs left over
        const int tt = t - p.pair_body;
        int pos;
        if (!p.pair_pack) {  // both tasks of pair pos: positions pos (light) and pos + half (heavy)
          const int half = p.pair_split_tail ? p.pair_r : G;
          light = tt < half;
          pos = light ? tt : tt - half;
        } else {  // heavy tasks on CTAs 0 .. r-1, light ones dealt over the other CTAs
          const int w = FAST ? fdiv(tt, p.fd_grid) : tt / G;
          const int c = tt - w * G;
          light = c >= p.pair_r;
          pos = light ? w * (G - p.pair_r) + (c - p.pair_r) : (w > 0 ? p.pair_r : c);
        }
        if (pos >= p.pair_r) {  // an empty entry: no rows, no keys
          k.b = 0, k.g = 0, k.mb = 0, k.kvh = 0;
          k.sq = p.Sq, k.kend = p.Sk, k.kshift = p.Sk - p.Sq, k.q_row0 = 0, k.k_row0 = 0, k.bc = 0;
          k.split = 0, k.ksplit = 0, k.nmax = 0;
          k.pos0[0] = k.pos0[1] = p.Sq;
          k.n[0] = k.n[1] = 0;
          return k;
        }
        t = p.pair_body / 2 + pos;
      }
    }
    const int units = p.B * p.groups;
    const int Mh = p.heavy_levels;
    if (PAIR && p.pair_grid > 0 && p.pair_nt > 0) {  // pair t; levels q0 .. q0+nt-1 go after all others
      const int Mm = Mh - p.pair_nt;
      const int n_main = units * Mm;
      int q;
      if (t < n_main) {  // L2 sections over the other levels
        const int su = p.section_units;
        const int section = FAST ? fdiv(t, p.fd_section_main) : t / (su * Mm);
        const int first_unit = section * su;
        int in_section = units - first_unit;
        if (in_section > su) in_section = su;
        const int idx = t - section * su * Mm;
        const int qq = FAST ? fdiv(idx, in_section == su ? p.fd_su : p.fd_last) : idx / in_section;
        unit = first_unit + (idx - qq * in_section);
        q = qq < p.pair_q0 ? qq : qq + p.pair_nt;
      } else {  // the left-over levels, level-major over all units
        const int k = t - n_main;
        const int lv = FAST ? fdiv(k, p.fd_units) : k / units;
        unit = k - lv * units;
        q = p.pair_q0 + lv;
      }
      mb = M - 1 - q;
    } else if (t < units * Mh) {  // heavier half: L2 sections, m_block decreasing inside each
      const int su = p.section_units;
      const int section = FAST ? fdiv(t, p.fd_section) : t / (su * Mh);
      const int first_unit = section * su;
      int in_section = units - first_unit;
      if (in_section > su) in_section = su;  // below su only in the last section
      const int idx = t - section * su * Mh;
      const int q = FAST ? fdiv(idx, in_section == su ? p.fd_su : p.fd_last) : idx / in_section;
      mb = M - 1 - q;
      unit = first_unit + (idx - q * in_section);
    } else {  // lighter half: one level (m_block) at a time over all units
      const int idx = t - units * Mh;
      const int q = FAST ? fdiv(idx, p.fd_units) : idx / units;
      mb = M - 1 - Mh - q;
      unit = idx - q * units;
    }
    if (light) mb = M - 1 - mb;
  }
  k.b = FAST ? fdiv(unit, p.fd_groups) : unit / p.groups;
  k.g = unit - k.b * p.groups;
  k.mb = mb;
  k.kvh = FAST ? fdiv(k.g * p.pack, p.fd_ratio) : (k.g * p.pack) / p.ratio;
  k.sq = p.Sq, k.kend = p.Sk, k.kshift = p.Sk - p.Sq, k.q_row0 = 0, k.k_row0 = 0, k.bc = k.b, k.split = 0;
  k.ksplit = 0;
  k.nmax = 0;
  if (tail_tile >= 0) {  // one tile, its key blocks halved over the two stages
    const int pos0 = (2 * k.mb + tail_tile) * p.pos_per_tile;
    const int nb = tile_blocks_len(p.Sq, p.Sk, p.Sk - p.Sq, 0, p.pos_per_tile, pos0);
    k.pos0[0] = k.pos0[1] = pos0;
    k.n[0] = (nb + 1) / 2;
    k.n[1] = nb - k.n[0];
    k.nmax = k.n[0];
    k.ksplit = k.n[1] > 0 ? k.n[0] : 0;
    if (k.ksplit == 0) k.n[1] = 0;
    return k;
  }
  for (int s = 0; s < 2; ++s) {
    k.pos0[s] = (2 * k.mb + s) * p.pos_per_tile;
    k.n[s] = tile_blocks_len(p.Sq, p.Sk, p.Sk - p.Sq, causal ? 1 : 0, p.pos_per_tile, k.pos0[s]);
    if (k.n[s] > k.nmax) k.nmax = k.n[s];
  }
  return k;
}

FA_HD Task decode_task(const Problem& p, int t) { return decode_task_k<-1, true>(p, t); }

// Does K/V block j need the element mask for a tile starting at pos0?  (the
// sequence tail, or the causal diagonal)
FA_HD bool block_needs_mask_len(int kend, int kshift, int causal, int pos0, int j) {
  const int64_t key_hi = static_cast<int64_t>(j) * kBN + kBN - 1;
  if (key_hi >= kend) return true;
  return causal && key_hi > static_cast<int64_t>(pos0) + kshift;
}

FA_HD bool block_needs_mask(const Problem& p, int pos0, int j) {
  return block_needs_mask_len(p.Sk, p.Sk - p.Sq, p.causal, pos0, j);
}

// The first K/V block that needs the mask (every later one needs it too):
// the tail starts at block kend / kBN; under the causal mask block j hides a
// key of the tile once j * kBN + kBN - 1 > pos0 + kshift.
FA_HD int first_masked_block(int kend, int kshift, int causal, int pos0) {
  int j = kend / kBN;
  if (causal) {
    const int64_t c1 = static_cast<int64_t>(pos0) + kshift + 1;
    const int jc = c1 > 0 ? static_cast<int>(c1 / kBN) : 0;
    if (jc < j) j = jc;
  }
  return j;
}

// Task t of a split-KV problem: t = ((b * groups + g) * splits + split) * M + m.
FA_HD Task decode_split_task(const Problem& p, int t) {
  Task k;
  const int M = p.mblocks;
  const int unit_split = fdiv(t, p.fd_mblocks);
  k.mb = t - unit_split * M;
  const int unit = fdiv(unit_split, p.fd_splits);
  k.split = unit_split - unit * p.splits;
  k.b = fdiv(unit, p.fd_groups);
  k.g = unit - k.b * p.groups;
  k.kvh = fdiv(k.g * p.pack, p.fd_ratio);
  const int k0 = k.split * p.split_blocks * kBN;
  int k1 = k0 + p.split_blocks * kBN;
  if (k1 > p.Sk) k1 = p.Sk;
  k.sq = p.Sq, k.kend = k1 - k0, k.kshift = p.Sk - p.Sq - k0;
  k.q_row0 = 0, k.k_row0 = k0, k.bc = k.b;
  k.ksplit = 0;
  k.nmax = 0;
  for (int s = 0; s < 2; ++s) {
    k.pos0[s] = (2 * k.mb + s) * p.pos_per_tile;
    k.n[s] = tile_blocks_len(k.sq, k.kend, k.kshift, p.causal, p.pos_per_tile, k.pos0[s]);
    if (k.n[s] > k.nmax) k.nmax = k.n[s];
  }
  return k;
}

// Split count for a problem whose (b, g, m_block) tasks may not fill `sms`
// persistent CTAs: 1 when they do (or the keys are few); otherwise the count
// that minimises the modelled time waves * (blocks per range + kSplitTaskCost):
// a range costs its K/V blocks plus a fixed start-up worth about five block
// times (the first tiles' HBM latency, the pipeline fill, the partial-result
// epilogue; fitted to GB300 timings of the decode workloads), at least 4
// blocks (512 keys) per range, at most 128 ranges.  Returns a count that
// leaves no range empty.
constexpr int kSplitTaskCost = 5;

FA_HD int choose_splits(const Problem& p, int sms) {
  const int64_t units = static_cast<int64_t>(p.B) * p.groups * p.mblocks;
  if (sms < 1 || units >= sms || p.kv_blocks < 8) return 1;
  int max_splits = p.kv_blocks / 4;
  if (max_splits > 128) max_splits = 128;
  int best = 1;
  int64_t best_cost = -1;
  for (int s = 1; s <= max_splits; ++s) {
    const int bps = ceil_div(p.kv_blocks, s);
    const int ranges = ceil_div(p.kv_blocks, bps);
    const int64_t tasks = units * ranges;
    const int64_t waves = (tasks + sms - 1) / sms;
    const int64_t cost = waves * (bps + kSplitTaskCost);
    if (best_cost < 0 || cost < best_cost) best_cost = cost, best = ranges;
  }
  return best;
}

// ---------------------------------------------------------------------------
// variable-length batches
// ---------------------------------------------------------------------------
// Upper bound on the tasks of any variable-length batch of `batch` sequences
// holding total_q queries: a sequence of sq queries has groups * ceil(sq * pack
// / 256) tasks, at most Hq * (sq / 256 + 1) whatever the pack.
FA_HD int64_t varlen_max_tasks(int batch, int heads_q, int64_t total_q) {
  return static_cast<int64_t>(heads_q) * ((total_q + 2 * kBM - 1) / (2 * kBM) + batch);
}

// Sort key of a sequence for the longest-first order: the K/V blocks of its
// heaviest tile.  Every tile of a non-causal sequence, and the last tile of a
// causal one (its last query sees key sk - 1), visits all ceil(sk / 128)
// blocks.  Sequences without queries have no tasks and sort last.
FA_HD int varlen_key(int sq, int sk) { return sq > 0 ? ceil_div(sk, kBN) : -1; }

// Sequence a comes before sequence b: larger key first, then lower index.
// Packed into one unsigned 64-bit value so that a descending sort of the
// values gives this order (index i is stored as ~i).
FA_HD uint64_t varlen_sort_value(int key, int index) {
  return (static_cast<uint64_t>(static_cast<uint32_t>(key + 1)) << 32) | static_cast<uint32_t>(~index);
}
FA_HD int varlen_sort_index(uint64_t value) { return static_cast<int>(~static_cast<uint32_t>(value)); }

// Tasks of one sequence: the fixed-length decomposition of a batch of one.
FA_HD Problem varlen_sequence_problem(const Problem& base, int sq, int sk, int d_qk, int d_v,
                                      int64_t l2_budget_bytes) {
  return make_problem_core(1, base.Hq, base.Hkv, sq, sk, d_qk, d_v, base.causal, l2_budget_bytes, base.pack);
}

// Record of the i-th task of sequence b (rows q_row0.., k_row0.. of the packed views).
FA_HD VarlenTask varlen_record(const Problem& seq, int b, int q_row0, int k_row0, int i) {
  const Task t = decode_task_k<-1, false, false, false>(seq, i);
  VarlenTask r;
  r.b = b, r.g = t.g, r.mb = t.mb, r.reserved = 0;
  r.q_row0 = q_row0, r.sq = seq.Sq, r.k_row0 = k_row0, r.sk = seq.Sk;
  return r;
}

// The task the kernel runs for a record.
template <bool FAST = false>
FA_HD Task task_from_record(const Problem& p, const VarlenTask& r) {
  Task k;
  k.b = r.b, k.g = r.g, k.mb = r.mb;
  k.kvh = FAST ? fdiv(k.g * p.pack, p.fd_ratio) : (k.g * p.pack) / p.ratio;
  k.sq = r.sq, k.kend = r.sk, k.kshift = r.sk - r.sq, k.q_row0 = r.q_row0, k.k_row0 = r.k_row0, k.bc = 0;
  k.split = 0;
  k.ksplit = 0;
  k.nmax = 0;
  for (int s = 0; s < 2; ++s) {
    k.pos0[s] = (2 * k.mb + s) * p.pos_per_tile;
    k.n[s] = tile_blocks_len(r.sq, r.sk, r.sk - r.sq, p.causal, p.pos_per_tile, k.pos0[s]);
    if (k.n[s] > k.nmax) k.nmax = k.n[s];
  }
  return k;
}

}  // namespace fa
