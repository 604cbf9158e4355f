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
//  * Task order: linear for the non-causal case (uniform cost); for the causal
//    case longest-processing-time first (m_blocks in decreasing order) inside
//    sections of `section_units` (b, g) units whose K/V fit in L2 together.
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
  int64_t num_tasks;  // B * groups * mblocks
};

struct Task {
  int b, g, mb;
  int kvh;       // K/V head read by this task
  int pos0[2];   // first sequence position of each stage's tile
  int n[2];      // K/V blocks each stage visits (0: nothing to do)
  int nmax;      // max(n[0], n[1])
};

FA_HD int ceil_div(int a, int b) { return (a + b - 1) / b; }

FA_HD int choose_pack(int Hq, int Hkv) {
  const int ratio = Hq / Hkv;
  return (ratio >= 1 && kBM % ratio == 0) ? ratio : 1;
}

// Fill the derived fields.  `pack_override` > 0 forces a pack (must divide
// both 128 and the ratio); l2_budget_bytes sizes the causal sections.
FA_HD Problem make_problem(int B, int Hq, int Hkv, int Sq, int Sk, int d_qk, int d_v, int causal,
                           int64_t l2_budget_bytes, int pack_override) {
  Problem p;
  p.B = B, p.Hq = Hq, p.Hkv = Hkv, p.Sq = Sq, p.Sk = Sk, p.causal = causal;
  p.ratio = Hq / Hkv;
  p.pack = pack_override > 0 ? pack_override : choose_pack(Hq, Hkv);
  p.groups = Hq / p.pack;
  p.pos_per_tile = kBM / p.pack;
  p.tiles = ceil_div(Sq, p.pos_per_tile);
  p.mblocks = ceil_div(p.tiles, 2);
  p.kv_blocks = ceil_div(Sk, kBN);
  p.num_tasks = static_cast<int64_t>(B) * p.groups * p.mblocks;
  // K/V bytes one (b, g) unit streams; units that share a KV head (pack = 1
  // with GQA) share those bytes in L2, which only makes the estimate safe.
  const int64_t kv_bytes = static_cast<int64_t>(Sk) * (d_qk + d_v) * 2;
  int64_t su = kv_bytes > 0 ? l2_budget_bytes / kv_bytes : 1;
  const int64_t units = static_cast<int64_t>(B) * p.groups;
  if (su < 1) su = 1;
  if (su > units) su = units > 0 ? units : 1;
  p.section_units = static_cast<int>(su);
  return p;
}

// K/V blocks a Q tile starting at pos0 visits.
FA_HD int tile_blocks(const Problem& p, int pos0) {
  if (pos0 >= p.Sq || p.kv_blocks == 0) return 0;
  if (!p.causal) return p.kv_blocks;
  int last = pos0 + p.pos_per_tile;
  if (last > p.Sq) last = p.Sq;
  const int64_t max_key = static_cast<int64_t>(last - 1) + p.Sk - p.Sq;
  if (max_key < 0) return 0;
  const int64_t n = max_key / kBN + 1;
  return n < p.kv_blocks ? static_cast<int>(n) : p.kv_blocks;
}

// Task t (0 <= t < num_tasks < 2^31; the host refuses larger problems).
FA_HD Task decode_task(const Problem& p, int t) {
  Task k;
  const int M = p.mblocks;
  int unit, mb;
  if (!p.causal) {
    unit = t / M;
    mb = t - unit * M;
  } else {
    const int su = p.section_units;
    const int units = p.B * p.groups;
    const int section = t / (su * M);
    const int first_unit = section * su;
    int in_section = units - first_unit;
    if (in_section > su) in_section = su;
    const int idx = t - section * su * M;
    const int q = idx / in_section;
    mb = M - 1 - q;  // heaviest m_block first
    unit = first_unit + (idx - q * in_section);
  }
  k.b = unit / p.groups;
  k.g = unit - k.b * p.groups;
  k.mb = mb;
  k.kvh = (k.g * p.pack) / p.ratio;
  k.nmax = 0;
  for (int s = 0; s < 2; ++s) {
    k.pos0[s] = (2 * k.mb + s) * p.pos_per_tile;
    k.n[s] = tile_blocks(p, k.pos0[s]);
    if (k.n[s] > k.nmax) k.nmax = k.n[s];
  }
  return k;
}

// Does K/V block j need the element mask for a tile starting at pos0?  (the
// sequence tail, or the causal diagonal)
FA_HD bool block_needs_mask(const Problem& p, int pos0, int j) {
  const int64_t key_hi = static_cast<int64_t>(j) * kBN + kBN - 1;
  if (key_hi >= p.Sk) return true;
  return p.causal && key_hi > static_cast<int64_t>(pos0) + p.Sk - p.Sq;
}

}  // namespace fa
