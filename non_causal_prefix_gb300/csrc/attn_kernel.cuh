// The attention kernel: work items, the per-tile online softmax and the
// warp-specialised persistent kernel (TMA loader, tcgen05 issuer, softmax /
// correction / epilogue warps).  Included once, by attn_fwd.cu, which holds
// the host side and the C ABI.
#pragma once

#include "sm103_ptx.cuh"

namespace ncp {

constexpr int BM = 128;                  // query rows per tile (one TMEM lane each)
constexpr int BN = 128;                  // keys per KV tile
constexpr int PRODUCER_WARP = 8;
constexpr int MMA_WARP = 9;
// D = 64 (P in TMEM columns of its own): a second MMA warp issues query tile
// 1's MMAs, so that neither tile's next S waits behind the other's P V.
constexpr int MMA_WARP2 = 10;
constexpr uint32_t TMEM_COLS = 512;
constexpr int MAX_SLOTS = 8;
// Block-causal form: per-CTA table of the image ids in each 128-token tile
// (min, max and "one image only"), held in shared memory; N <= 128 * this.
constexpr int MAX_SEQ_TILES = 1024;
// Split tail (see schedule_item): most pieces one merge reads (plus one for a
// range boundary), least key tiles per tail CTA (a piece pays a Q load, a
// pipeline fill and a partial write + merge), and most tail units (units in
// a last, partly filled round: fewer than the SM count).
constexpr int MAX_PIECES = 8;
constexpr int MIN_PIECE_TILES = 4;
constexpr int MAX_TAIL_UNITS = 1024;
// Dense forms: most CTAs sharing a tail (their range bounds travel in the
// kernel parameters).
constexpr int MAX_TAIL_CTAS = 256;
// Masked forms: most query pairs (256-row units along the sequence).
constexpr int MAX_Q_PAIRS = MAX_SEQ_TILES / 2;
// Rescale O only when the running row maximum (log2 units) grows by more than
// this; otherwise keep the stale maximum.  Exact, because the final 1/l uses
// the same maximum as the accumulated O, and p <= 2^8 stays far from overflow.
constexpr float RESCALE_THRESHOLD = 8.0f;

// Polynomial share of the exponentials (compile-time; overridable with -D).
#ifndef NCP_POLY_NUM_D128
#define NCP_POLY_NUM_D128 0
#endif
#ifndef NCP_POLY_DEN_D128
#define NCP_POLY_DEN_D128 4
#endif
#ifndef NCP_POLY_NUM_D64
#define NCP_POLY_NUM_D64 0
#endif
#ifndef NCP_POLY_DEN_D64
#define NCP_POLY_DEN_D64 4
#endif
// D = 64: P in TMEM columns of its own (1) or over S (0); see Cfg::P_OWN.
#ifndef NCP_P_OWN
#define NCP_P_OWN 1
#endif

template <int D>
struct Cfg {
  static constexpr int CHUNKS = D / 64;                  // 128-byte swizzle columns per row
  // TMEM columns (512) of S_i, P_i and O_i for query tile i.  D = 128: S_0,
  // S_1, O_0, O_1 take 128 each, and P_i (bf16, two per column) is written
  // over the first 64 columns of S_i, so S_i(j + 1) follows the P V that
  // reads P_i(j).  D = 64: O_i takes 64 columns, which leaves 64 for each P_i
  // (P_OWN), and S_i(j + 1) is issued as soon as the softmax warps have read
  // S_i(j) into registers, so that it runs during their softmax: a query
  // tile's key step is then about its softmax, not softmax + P V + S.
  static constexpr bool P_OWN = (D == 64) && NCP_P_OWN;
  __host__ __device__ static constexpr uint32_t s_col(int i) { return 128u * i; }
  __host__ __device__ static constexpr uint32_t p_col(int i) { return P_OWN ? 256u + 64u * i : 128u * i; }
  __host__ __device__ static constexpr uint32_t o_col(int i) { return P_OWN ? 384u + 64u * i : 256u + 128u * i; }
  static constexpr uint32_t TILE_BYTES = BN * D * 2;     // one K or V tile; one Q tile (BM == BN)
  static constexpr uint32_t CHUNK_BYTES = BN * 128;      // 128 rows x 128 bytes
  // K/V ring, in tile-sized slots (paired into entries below).  D = 64: 6
  // rather than 8 (measured as fast or faster on every D = 64 workload): the
  // 32 KB less shared memory leaves a larger L1 for the register spills of
  // the 11-warp kernel.
  static constexpr int NSLOT = (D == 128) ? 4 : 6;
  static constexpr uint32_t RING_OFF = 0;
  // The ring holds NSLOT / 2 entries of two tiles (K half, then V half), one
  // full barrier expecting both loads and one release each.  D = 64
  // (KV_PAIRS): a key tile's K and V.  D = 128: K of a key tile and V of the
  // item's previous visited key tile (S_i(j) and P_i V(j - 1) are issued
  // together), an item's first entry holding K alone and an entry after its
  // last key tile holding the last V alone.
  static constexpr bool KV_PAIRS = P_OWN;
  static constexpr int NRING = NSLOT / 2;
  static constexpr uint32_t ENTRY_BYTES = 2 * TILE_BYTES;
  static_assert(NSLOT % 2 == 0, "ring entries take two slots each");
  static constexpr uint32_t Q_OFF = RING_OFF + NSLOT * TILE_BYTES;
  static constexpr uint32_t BAR_OFF = Q_OFF + 2 * TILE_BYTES;
  static constexpr uint32_t SMEM_BYTES = BAR_OFF + 512 + 1024;  // barriers + 1 KiB alignment slack
  static constexpr uint32_t SUM_OFF = BAR_OFF + 512;             // masked forms: tile table
  static constexpr uint32_t TAIL_OFF = SUM_OFF + 3 * 4 * MAX_SEQ_TILES;  // and tail prefix sums
  static constexpr uint32_t ITEMS_OFF = TAIL_OFF + 4 * (MAX_TAIL_UNITS + 4);  // and tail items
  static constexpr uint32_t ORDER_OFF = ITEMS_OFF + 48 * 32;  // and the unit order tables
  // and, per work-item slot, bit masks over the key tiles: visited by the
  // item's query pair, and seen whole by query tile 0 / by query tile 1
  static constexpr uint32_t MASK_OFF = ORDER_OFF + 4 * (3 * MAX_Q_PAIRS + 2);
  static constexpr int MASK_WORDS = MAX_SEQ_TILES / 32;
  static constexpr uint32_t SMEM_BYTES_BC = MASK_OFF + 2 * 3 * 4 * MASK_WORDS + 1024;
  // Share of the exponentials computed by the FMA-pipe polynomial instead of
  // the MUFU unit: POLY_NUM of every POLY_DEN packed pairs.  On GB300 the
  // MUFU unit does about 30 exp2 per clock per SM and the polynomial about 13:
  // every measured share above 0 was slower, so the default is 0.
  static constexpr int POLY_NUM = (D == 128) ? NCP_POLY_NUM_D128 : NCP_POLY_NUM_D64;
  static constexpr int POLY_DEN = (D == 128) ? NCP_POLY_DEN_D128 : NCP_POLY_DEN_D64;
  static_assert(POLY_DEN >= 1 && POLY_NUM >= 0 && POLY_NUM <= POLY_DEN, "polynomial share");
  __host__ __device__ static constexpr bool poly_pair(int c) { return (c % POLY_DEN) >= POLY_DEN - POLY_NUM; }
};

// Threads of a CTA: 10 warps (8 softmax, the loader, the MMA warp), plus the
// second MMA warp where P has columns of its own.
template <int D>
__host__ __device__ constexpr int num_threads() {
  return Cfg<D>::P_OWN ? 352 : 320;
}

struct SharedCtl {
  uint64_t q_full;
  uint64_t q_free;
  uint64_t kv_full[MAX_SLOTS];   // per K/V ring entry (Cfg::NRING of them are used)
  uint64_t kv_empty[MAX_SLOTS];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_full[2];
  uint64_t o_free[2];
  uint64_t pv_done[2];     // D = 64: a P V of query tile i, not an item's last, is complete
  uint64_t s_free[2];      // D = 64: the 4 softmax warps of query tile i have read S_i
  uint64_t part_done[2];   // the 4 warps of a query tile wrote their partial rows
  uint64_t merge_ready[2]; // the piece's arrival count is known (SharedCtl::last)
  uint64_t drain;
  uint64_t tail_ready;     // masked forms: this CTA's tail items are in shared memory
  uint64_t item_full[2];   // the loader has written work item slot s (item n: slot n & 1)
  uint64_t item_empty[2];  // every warp but the loader is done with slot s's item
  int last[2];             // this piece is the last of its unit: merge and store
  int n_tail_items;        // masked forms: tail items of this CTA kept in shared memory
  uint32_t tmem_base;
  int abort_flag;
  // Work items as the loader decoded them, two slots (an Item, 48 bytes at
  // most): the other roles read them instead of decoding each item again.
  alignas(16) unsigned char item_ring[2][48];
};
static_assert(sizeof(SharedCtl) <= 512, "the barrier block holds 512 bytes");

// Work schedule of one launch.  Units are (b, h, pair of 128-row query
// tiles), n_units = B * H * q_pairs of them; see schedule_item.
struct Sched {
  int n_units;
  int q_pairs;     // ceil(Nq / unit_rows): units per (b, h); query block fastest
  int H, Nq;
  int unit_rows;   // query rows per unit: two 128-row tiles
  int n_whole;     // units walked whole
  int tail_units;  // units after them, cut into key ranges (0: none)
  int tail_ctas;   // CTAs sharing the tail (0: no tail)
  // Dense forms with short key sequences (see make_sched): the loader
  // prefetches each next work item's Q into L2.
  int prefetch_q;
  // Dense forms: CTA c of the tail holds tail tiles [bounds[c], bounds[c + 1])
  // (tiles of the tail units in unit order), every range non-empty.
  int bounds[MAX_TAIL_CTAS + 1];
};

struct Params {
  CUtensorMap tm_q;
  CUtensorMap tm_k[2];   // [0] prefix segment, [1] current segment
  CUtensorMap tm_v[2];
  __nv_bfloat16* out;
  // Masked forms (block-causal, masked prefix-cached): image id per key
  // position [Np + Nq] (-1 = text) and, optionally, key_valid [B, Np + Nq]
  // (nullptr: every key valid).  Query i sits at position Np + i.
  const int* image_ids;
  const unsigned char* key_valid;
  int Nq, H;
  Sched sc;
  float* ws_part;          // [piece slot][query tile][D / 4 + 1][128 rows][4]: O, then m, l
  // [tail unit][query tile] arrival counters: (epoch << 32) | pieces counted
  // in.  A counter whose epoch is not this launch's counts as 0, so a launch
  // that gave up part-way leaves nothing behind for the next one.
  unsigned long long* ws_count;
  unsigned int epoch;      // this launch's tag (never 0: a cleared counter is no launch's)
  int n_tok[2];          // tokens per key segment
  int n_tiles[2];        // KV tiles per key segment
  float scale_log2;      // D^-0.5 * log2(e)
  int fault_mode;
  unsigned long long wait_limit_ns;
};

// ----------------------------------------------------------------------------
// Work units and items
// ----------------------------------------------------------------------------
struct Unit {
  int b, h, q0;
  bool two;  // the second 128-row query tile has at least one row
};

// Masked forms: the order of the units.  A unit's work depends only on its
// query pair (the same for every batch and head): its cost, bc_pair_tile_cost
// summed over the key tiles, orders the query pairs, most first (ties: the
// later pair first); pairs of one cost form a level.  Units go level by level, and
// within a level head-major with the query pair fastest, as in the dense
// order, so that the CTAs running at one time share few heads' K/V in L2.
// Tables (int block): [0] number of levels L, [1 .. L + 1] first index into
// qp_order of each level (then q_pairs), then qp_order[q_pairs] at
// ORDER_QP = 2 + MAX_Q_PAIRS.
struct UnitOrder {
  const int* tab;
};
constexpr int ORDER_QP = 2 + MAX_Q_PAIRS;

// Position of query pair q in the unit order, from the visited-tile counts
// of the q_pairs pairs: more tiles first, the later pair first among equals.
__host__ __device__ __forceinline__ int order_rank(const int* cnt, int q_pairs, int q) {
  int rank = 0;
  const int cq = cnt[q];
  for (int q2 = 0; q2 < q_pairs; ++q2) rank += (cnt[q2] > cq || (cnt[q2] == cq && q2 > q)) ? 1 : 0;
  return rank;
}

// The levels of the order table `ob` once its qp_order is filled (one thread).
__host__ __device__ __forceinline__ void order_levels(int* ob, const int* cnt, int q_pairs) {
  int n_lvl = 0;
  for (int r = 0; r < q_pairs; ++r)
    if (r == 0 || cnt[ob[ORDER_QP + r]] != cnt[ob[ORDER_QP + r - 1]]) ob[1 + n_lvl++] = r;
  ob[1 + n_lvl] = q_pairs;
  ob[0] = n_lvl;
}

__host__ __device__ __forceinline__ Unit decode_unit(const Sched& s, bool bc, int unit,
                                                     const UnitOrder* ord = nullptr) {
  Unit u;
  // Dense forms: query pair fastest, so the CTAs running at one time share
  // the K/V of a few heads in L2.  Masked forms: by levels of work (above).
  const int n_bh = s.n_units / s.q_pairs;  // B * H
  int qp, bh;
  if (bc) {
    const int* lvl = ord->tab + 1;
    int a = 0, b = ord->tab[0] - 1;  // the level holding this unit
    while (a < b) {
      const int mid = (a + b + 1) / 2;
      if (lvl[mid] * n_bh <= unit) a = mid; else b = mid - 1;
    }
    const int len = lvl[a + 1] - lvl[a];
    const int w = unit - lvl[a] * n_bh;
    bh = w / len;
    qp = ord->tab[ORDER_QP + lvl[a] + w % len];
  } else {
    qp = unit % s.q_pairs;
    bh = unit / s.q_pairs;
  }
  u.h = bh % s.H;
  u.b = bh / s.H;
  u.q0 = qp * s.unit_rows;
  u.two = (u.q0 + s.unit_rows / 2) < s.Nq;
  return u;
}

struct Item {
  Unit u;
  int t_begin, t_end;  // key tiles [t_begin, t_end) of the concatenated key sequence
  int tail;            // -1: a whole unit; else the tail unit this piece belongs to
  int piece, pieces;   // this piece's index among the tail unit's pieces, and their count
  int slot0;           // workspace slot of the tail unit's piece 0 (piece k: slot0 + k)
};

// Block-causal visibility (definition prefix_cached_block_causal_h32_d128_
// prefix0): query i sees key j iff j <= i, or both carry the same image id >= 0.
// Tiles are summarised by the range [lo, hi] of their non-negative ids (lo >
// hi: text only) and by `uni` (every token in one image).
// The three arrays sit back to back in shared memory (MAX_SEQ_TILES each),
// reached from one base to keep the loops' live state small.
struct TileTable {
  const int* base;
  __host__ __device__ __forceinline__ int lo(int t) const { return base[t]; }
  __host__ __device__ __forceinline__ int hi(int t) const { return base[MAX_SEQ_TILES + t]; }
  __host__ __device__ __forceinline__ int uni(int t) const { return base[2 * MAX_SEQ_TILES + t]; }
};

// Key tiles walk the prefix segment (tiles [0, T0)) then the current one;
// position of the first key of tile t, and its number of keys.
__host__ __device__ __forceinline__ int key_tile_pos(const Params& p, int t) {
  const int T0 = p.n_tiles[0];
  return t < T0 ? t * BN : p.n_tok[0] + (t - T0) * BN;
}
__host__ __device__ __forceinline__ int key_tile_len(const Params& p, int t) {
  const int T0 = p.n_tiles[0];
  const int seg = t < T0 ? 0 : 1;
  return min(BN, p.n_tok[seg] - (t - (seg ? T0 : 0)) * BN);
}

// Some query row of the unit sees some key of tile t: causally (the tile
// starts at or before the unit's last row, at position Np + row), or through
// an image id both may share (their id ranges meet; the query tiles are the
// current segment's tiles T0 + qt).  key_valid only removes keys, so the
// filter stays exact: a skipped tile has no visible pair.
__host__ __device__ __forceinline__ bool bc_unit_visits(const TileTable& tt, const Params& p,
                                                        const Unit& u, int t) {
  const int r_last = p.n_tok[0] + min(u.q0 + 2 * BM, p.Nq) - 1;
  if (key_tile_pos(p, t) <= r_last) return true;
  const int qt0 = p.n_tiles[0] + u.q0 / BM;
  const int qt1 = u.two ? qt0 + 1 : qt0;
  const int qlo = min(tt.lo(qt0), tt.lo(qt1));
  const int qhi = max(tt.hi(qt0), tt.hi(qt1));
  return qlo <= tt.hi(t) && tt.lo(t) <= qhi;
}

// Every query row of query tile qt (current-segment tile T0 + qt, first row
// q_first) sees every key of tile t through causality or one shared image
// (key_valid aside): the keys all precede the rows, or both tiles hold one
// and the same image.
__host__ __device__ __forceinline__ bool bc_tile_full(const TileTable& tt, const Params& p,
                                                      int qt, int q_first, int t) {
  if (key_tile_pos(p, t) + key_tile_len(p, t) - 1 <= p.n_tok[0] + q_first) return true;
  const int tq = p.n_tiles[0] + qt;
  return tt.uni(tq) && tt.uni(t) && tt.lo(tq) == tt.lo(t);
}

// Cost of key tile t to the query pair of unit u (masked forms), in units of
// about 1/16 us of a GB300 CTA: 0 if no row of the pair sees the tile, else
// 26 for a pair of two query tiles or 22 for one (one tile loses the other's
// overlap), plus 6 for each query tile that sees only part of the key tile
// (it builds a row mask).  Fitted to the per-CTA times of a traced
// block-causal launch: 1.62, 1.38 and 0.35 us.  Only the order of the units
// uses it.
__host__ __device__ __forceinline__ int bc_pair_tile_cost(const TileTable& tt, const Params& p,
                                                          const Unit& u, int t) {
  if (!bc_unit_visits(tt, p, u, t)) return 0;
  const int qt0 = u.q0 / BM;
  int c = u.two ? 26 : 22;
  if (!bc_tile_full(tt, p, qt0, u.q0, t)) c += 6;
  if (u.two && !bc_tile_full(tt, p, qt0 + 1, u.q0 + BM, t)) c += 6;
  return c;
}

// Owner of tail position x (tail positions in unit order): CTA c of G holds
// positions [c W / G, (c + 1) W / G).
__host__ __device__ __forceinline__ long long tail_owner(long long x, long long W, long long G) {
  return ((x + 1) * G - 1) / W;
}

// Summary of the image ids of key tile t of the masked forms (see TileTable),
// one thread's version (the kernel builds its table warp by warp).
__host__ __device__ inline void tile_summary(const Params& p, const int* ids, int t, int& lo,
                                             int& hi, int& uni) {
  lo = 0x7fffffff;
  hi = -1;
  bool text = false;
  const int pos0 = key_tile_pos(p, t), len = key_tile_len(p, t);
  for (int e = 0; e < len; ++e) {
    const int id = ids[pos0 + e];
    if (id < 0) {
      text = true;
    } else {
      lo = id < lo ? id : lo;
      hi = id > hi ? id : hi;
    }
  }
  uni = (!text && lo == hi) ? 1 : 0;
}

// Masked forms' tail: the key-tile table, and pre[r] = key tiles visited by
// the tail units before tail unit r (pre[tail_units]: all of them).
// items[0 .. n_items) (kernel only): this CTA's first tail items, worked out
// once at the start of the kernel.
struct MaskedTail {
  const Params* p;
  TileTable tt;
  const int* pre;
  const Item* items;
  int n_items;
  UnitOrder ord;
};

// Most tail items of one CTA kept in shared memory (later ones, rare, are
// worked out when reached).  Overridable with -D to test that path.
#ifndef NCP_MAX_CTA_TAIL_ITEMS
#define NCP_MAX_CTA_TAIL_ITEMS 32
#endif
constexpr int MAX_CTA_TAIL_ITEMS = NCP_MAX_CTA_TAIL_ITEMS;
static_assert(MAX_CTA_TAIL_ITEMS >= 1 && MAX_CTA_TAIL_ITEMS <= 32, "tail item list: 1 to 32 items");
static_assert(sizeof(Item) <= 48, "tail item list: 48 bytes per item in shared memory");

// Masked forms' tail: the cost of one tail item, in visited key tiles, over
// and above its tiles (a Q load, a pipeline fill and an epilogue; for a piece
// also the partial write and count-in).  Charged once per tail unit, at the
// unit's start: a CTA whose range takes in many small units, or crosses into
// a second unit, gets correspondingly fewer tiles.  Overridable with -D.
#ifndef NCP_MASKED_UNIT_COST
#define NCP_MASKED_UNIT_COST 3
#endif
constexpr int MASKED_UNIT_COST = NCP_MASKED_UNIT_COST;
static_assert(MASKED_UNIT_COST >= 0, "masked tail unit cost");

// CTAs sharing a masked tail of W visited tiles: at most the launch's
// tail_ctas, and at least MIN_PIECE_TILES visited tiles each.
__host__ __device__ __forceinline__ long long masked_tail_ctas(const Sched& s, long long W) {
  long long G = W / MIN_PIECE_TILES;
  if (G > s.tail_ctas) G = s.tail_ctas;
  return G < 1 ? 1 : G;
}

// Fill `it` with the tail piece of tail unit r that covers tail positions
// [lo, hi) clipped to the unit's [u0, u1); owner(x) is the CTA holding tail
// position x.  to_tile maps a position inside the unit to its key tile
// (identity for the dense forms).
template <class Owner, class ToTile>
__host__ __device__ __forceinline__ void tail_piece(const Sched& s, bool bc, int c, long long r,
                                                    long long lo, long long hi, long long u0,
                                                    long long u1, Owner owner, ToTile to_tile,
                                                    const UnitOrder* ord, Item& it) {
  const long long first = owner(u0);
  const long long last = owner(u1 - 1);
  const int v0 = static_cast<int>((lo > u0 ? lo : u0) - u0);
  const int v1 = static_cast<int>((hi < u1 ? hi : u1) - u0);
  it.u = decode_unit(s, bc, s.n_whole + static_cast<int>(r), ord);
  it.t_begin = to_tile(it.u, v0);
  it.t_end = to_tile(it.u, v1 - 1) + 1;
  if (first == last) {  // the whole unit in one range: no merge
    it.tail = -1;
    it.piece = 0;
    it.pieces = 1;
    it.slot0 = 0;
  } else {
    it.tail = static_cast<int>(r);
    it.piece = c - static_cast<int>(first);
    it.pieces = static_cast<int>(last - first) + 1;
    it.slot0 = static_cast<int>(first + r);
  }
}

// Tail item j of CTA c of the masked forms (see schedule_item); to_tile(u,
// v) gives the v-th key tile unit u visits.
template <class ToTile>
__host__ __device__ __forceinline__ bool masked_tail_item(const Sched& s, const MaskedTail& mt,
                                                          int T, int c, int j, Item& it,
                                                          ToTile to_tile) {
  // Cost positions: tail unit r spans [P(r), P(r + 1)), P(r) = pre[r] + C r
  // with C = MASKED_UNIT_COST: C positions of item cost, then its visited
  // tiles.
  constexpr int C = MASKED_UNIT_COST;
  const int* pre = mt.pre;
  const long long G = masked_tail_ctas(s, pre[s.tail_units]);
  const long long W = pre[s.tail_units] + static_cast<long long>(C) * s.tail_units;
  if (c >= G) return false;
  const long long lo = c * W / G, hi = (c + 1) * W / G;
  if (lo >= hi) return false;
  // The tail unit holding position lo: the last r with P(r) <= lo (P rises
  // strictly: every unit visits its diagonal tiles).
  int a = 0, b = s.tail_units - 1;
  while (a < b) {
    const int mid = (a + b + 1) / 2;
    if (pre[mid] + C * mid <= lo) a = mid; else b = mid - 1;
  }
  // Item j: the j-th unit whose tiles meet [lo, hi).  Past the first, every
  // unit the range reaches does (its tiles follow its cost positions); the
  // first may be missed only when the range ends inside its cost positions.
  const int r = a + j;
  if (r >= s.tail_units || pre[r] + C * (r + 1) >= hi) return false;
  tail_piece(s, true, c, r, lo, hi, pre[r] + C * (r + 1), pre[r + 1] + C * (r + 1),
             [&](long long x) { return tail_owner(x, W, G); }, to_tile, &mt.ord, it);
  return true;
}

// Item n of CTA c in a grid of g, or false past its last one.
//
// No tail (s.tail_ctas == 0): CTA c takes units n g + c, round robin (masked
// forms: a snake, rounds alternating direction, so that a CTA that took a long
// unit in one round takes a short one in the next).
//
// Tail: the n_whole = rounds * g first units go the same way; the work of the
// tail_units units left is laid out in unit order as W tail positions and cut
// into G ranges, one per CTA c < G.  Dense forms: a position is a key tile,
// W = tail_units * T, and the ranges (s.bounds, chosen on the host) weigh each
// extra piece a CTA takes.  Masked forms (equal ranges of cost): each unit is
// MASKED_UNIT_COST positions of item cost, then one position per *visited*
// key tile (mt->pre counts them), G = masked_tail_ctas(visited tiles).  A range
// that crosses a unit boundary gives its CTA one piece of each unit.  Each
// piece leaves its partial (O, m, l) in workspace slot c + r (r: the tail
// unit), which is unique: a CTA later in the order only meets later units.
template <bool BC>
__host__ __device__ __forceinline__ bool schedule_item(const Sched& s, int T, int g, int c, int n,
                                                       Item& it, const MaskedTail* mt) {
  it.tail = -1;
  it.piece = 0;
  it.pieces = 1;
  it.slot0 = 0;
  it.t_begin = 0;
  it.t_end = T;
  const int rounds = s.tail_ctas ? s.n_whole / g : 0;
  if (s.tail_ctas == 0 || n < rounds) {
    const int unit = n * g + ((BC && (n & 1)) ? g - 1 - c : c);
    if (unit >= s.n_whole) return false;
    it.u = decode_unit(s, BC, unit, BC ? &mt->ord : nullptr);
    return true;
  }
  const int j = n - rounds;  // tail item of this CTA
  if (!BC) {
    const int G = s.tail_ctas;
    if (c >= G) return false;
    const long long lo = s.bounds[c], hi = s.bounds[c + 1];
    const long long r = lo / T + j;
    if (r >= s.tail_units || r * T >= hi) return false;
    auto owner = [&](long long x) {  // the last CTA whose range starts at or before x
      int a = 0, b = G - 1;
      while (a < b) {
        const int mid = (a + b + 1) / 2;
        if (s.bounds[mid] <= x) a = mid; else b = mid - 1;
      }
      return static_cast<long long>(a);
    };
    tail_piece(s, false, c, r, lo, hi, r * T, (r + 1) * T, owner,
               [](const Unit&, int v) { return v; }, nullptr, it);
    return true;
  }
  return masked_tail_item(s, *mt, T, c, j, it, [&](const Unit& u, int v) {
    int seen = 0;
    for (int t = 0; t < T; ++t)
      if (bc_unit_visits(mt->tt, *mt->p, u, t) && seen++ == v) return t;
    return T - 1;
  });
}

template <bool BC>
__device__ __forceinline__ bool get_item(const Params& p, const MaskedTail* mt, int T, int n,
                                         Item& it) {
  if (BC && p.sc.tail_ctas > 0) {
    const int j = n - p.sc.n_whole / static_cast<int>(gridDim.x);
    if (j >= 0 && j < mt->n_items) {
      it = mt->items[j];
      return true;
    }
    if (j >= 0 && j < MAX_CTA_TAIL_ITEMS) return false;  // the list holds every item
  }
  return schedule_item<BC>(p.sc, T, static_cast<int>(gridDim.x), static_cast<int>(blockIdx.x), n,
                           it, mt);
}

// Per-row mask of one key tile of the masked forms: key position c0 + c is
// visible to the query at position qi (image id idq) iff c0 + c <= qi or its
// id equals idq >= 0, and (with key_valid, batch b) the key is valid.  The
// id and flag pointers are formed from the kernel parameters where they are
// read, so that they are not live across the key loop.
struct RowMask {
  int c0, qi, idq, b;
  bool ids;    // test image ids (false: every key of the tile visible)
  bool valid;  // test key_valid (false: every key valid)
};

// Masked forms: this row's visibility of one key tile's 128 keys as a
// bitmask (masked: some key is hidden).  It reads only the image ids and
// key_valid, so the softmax warps build it while they wait for the tile's
// scores.
__device__ __forceinline__ void build_row_mask(const Params& p, const RowMask& mask,
                                               uint32_t (&vis)[4], bool& masked) {
  const int n_keys = p.n_tok[0] + p.n_tok[1];  // key positions (nothing past them is read)
  // The warp builds it together (the flags are warp-uniform): lane l reads the
  // ids and flags of keys l, 32 + l, 64 + l, 96 + l (coalesced), so that one
  // ballot per 32 keys gives a mask word in key order.
  vis[0] = vis[1] = vis[2] = vis[3] = ~0u;
  masked = false;
  const int lane = static_cast<int>(threadIdx.x & 31u);
  if (mask.ids) {
    masked = true;
    const int* ids = p.image_ids + mask.c0;
    int kid[4];  // keys past the last position read as text; `valid` masks them
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = 32 * e + lane;
      kid[e] = (mask.c0 + c < n_keys) ? __ldg(ids + c) : -1;
    }
    // Causal part: keys c <= qi - c0.
    const int lim = mask.qi - mask.c0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int d = lim - 32 * e;  // keys 32 e .. 32 e + d of this word
      vis[e] = d >= 31 ? ~0u : (d < 0 ? 0u : (2u << d) - 1u);
    }
    // Image part, once per distinct image id among the warp's rows.
    uint32_t pending = __ballot_sync(0xffffffffu, mask.idq >= 0);
    while (pending) {
      const int X = __shfl_sync(0xffffffffu, mask.idq, __ffs(pending) - 1);
      const bool mine = mask.idq == X;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t w = __ballot_sync(0xffffffffu, kid[e] == X);
        if (mine) vis[e] |= w;
      }
      pending &= ~__ballot_sync(0xffffffffu, mine);
    }
  }
  if (mask.valid) {
    // key_valid, the same for every row: keys past the last position count
    // as valid here (`valid` masks them).
    const unsigned char* kv = p.key_valid + static_cast<size_t>(mask.b) * n_keys + mask.c0;
    uint32_t okw[4];
    bool all = true;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = 32 * e + lane;
      okw[e] = __ballot_sync(0xffffffffu, mask.c0 + c >= n_keys || __ldg(kv + c) != 0);
      all = all && okw[e] == ~0u;
    }
    if (!all) {
      masked = true;
#pragma unroll
      for (int e = 0; e < 4; ++e) vis[e] &= okw[e];
    }
  }
}

// One 128-key tile of the online softmax for this thread's query row:
// S (fp32, TMEM) -> running max m and sum l (log2 domain) -> P (bf16) at
// p_addr (64 columns); O is rescaled in TMEM when m moved.  before_store()
// runs before P and O are written and returns false if they must not be (a
// wait gave up); the tile then stops there and returns false.
template <int D, bool BC, class AfterRead, class BeforeStore>
__device__ __forceinline__ bool softmax_tile(uint32_t s_addr, uint32_t p_addr, uint32_t o_addr,
                                             int valid, float sl2, bool may_rescale,
                                             const uint32_t (&vis)[4], bool masked, float& m,
                                             float& l, AfterRead after_read,
                                             BeforeStore before_store) {
  float s[BN];
  {
    uint32_t r[BN];
#pragma unroll
    for (int c = 0; c < BN; c += 32) tmem_ld32(s_addr + c, r + c);
    tmem_wait_ld();
    after_read();
#pragma unroll
    for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(r[c]);
  }
  if (valid < BN) {
#pragma unroll
    for (int c = 0; c < BN; ++c)
      if (c >= valid) s[c] = -INFINITY;
  }
  if (BC && masked) {
#pragma unroll
    for (int c = 0; c < BN; ++c)
      if (!((vis[c / 32] >> (c % 32)) & 1u)) s[c] = -INFINITY;
  }
  // Row maximum: four independent chains of 3-input max.
  float mx0 = fmax3(s[0], s[1], s[2]), mx1 = fmax3(s[3], s[4], s[5]);
  float mx2 = fmax3(s[6], s[7], s[8]), mx3 = fmax3(s[9], s[10], s[11]);
#pragma unroll
  for (int c = 12; c + 8 <= BN; c += 8) {
    mx0 = fmax3(mx0, s[c], s[c + 1]);
    mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
    mx2 = fmax3(mx2, s[c + 4], s[c + 5]);
    mx3 = fmax3(mx3, s[c + 6], s[c + 7]);
  }
  mx0 = fmax3(mx0, s[BN - 4], s[BN - 3]);
  mx1 = fmax3(mx1, s[BN - 2], s[BN - 1]);
  const float m_tile = fmax3(mx0, mx1, fmaxf(mx2, mx3)) * sl2;
  float alpha = 1.f;
  bool rescale = false;
  if (m_tile > m + RESCALE_THRESHOLD) {
    alpha = ex2(m - m_tile);
    l *= alpha;
    m = m_tile;
    rescale = may_rescale;
  }
  // p = 2^(s * scale * log2(e) - m) on packed pairs; pairs selected by
  // poly_pair go through the FMA-pipe polynomial, the rest through MUFU.
  const uint64_t sl2x2 = pk2(sl2, sl2);
  // A row with no visible key yet (block-causal form only) keeps m = -inf:
  // use 0 so that its masked scores give p = 0 instead of NaN.
  const float m_ref = (BC && m == -INFINITY) ? 0.f : m;
  const uint64_t neg_m2 = pk2(-m_ref, -m_ref);
  uint64_t acc0 = 0, acc1 = 0;  // two packed running sums (bits 0 = 0.0f)
  uint32_t pk[BN / 2];
#pragma unroll
  for (int c = 0; c < BN / 2; ++c) {
    const uint64_t x = ffma2(pk2(s[2 * c], s[2 * c + 1]), sl2x2, neg_m2);
    float p0, p1;
    if (Cfg<D>::poly_pair(c)) {
      exp2_poly2(x, p0, p1);
    } else {
      float x0, x1;
      up2(x, x0, x1);
      p0 = ex2(x0);
      p1 = ex2(x1);
    }
    if (c & 1)
      acc1 = fadd2(acc1, pk2(p0, p1));
    else
      acc0 = fadd2(acc0, pk2(p0, p1));
    pk[c] = pack_bf16x2(p0, p1);
  }
  {
    float a0, a1, a2, a3;
    up2(acc0, a0, a1);
    up2(acc1, a2, a3);
    l += (a0 + a1) + (a2 + a3);
  }
  if (!before_store()) return false;
  tmem_st32(p_addr + 0, pk);
  tmem_st32(p_addr + 32, pk + 32);
  if (__any_sync(0xffffffffu, rescale)) {
    // O holds the complete sum through the previous tile: D = 128, this S
    // was issued after the previous P V and its commit has fired; D = 64,
    // before_store() waited for that P V.  Rows of this warp that keep their
    // maximum scale by 1.
    const uint64_t alpha2 = pk2(alpha, alpha);
#pragma unroll
    for (int c = 0; c < D; c += 32) {
      uint32_t r[32];
      tmem_ld32(o_addr + c, r);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        float a0, a1;
        up2(fmul2(pk2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), alpha2), a0, a1);
        r[e] = __float_as_uint(a0);
        r[e + 1] = __float_as_uint(a1);
      }
      tmem_st32(o_addr + c, r);
    }
  }
  return true;
}

// Merge of a tail unit's pieces for one row: `part` points at this row's
// partial in piece 0's slot (piece k's is 2 (D / 4 + 1) 128 float4 further),
// D / 4 groups of O then (m, l) in the next group, group-major (128 float4
// apart).  Pieces are combined in piece order, so the result does not depend
// on which piece finished last: the common maximum and the sum first, then O
// in groups of 64 columns (16 loads in flight per piece), stored as bf16 to
// `dst` (nullptr: a padding row, nothing stored).  With OWN, the merging piece
// `own` takes its O from TMEM (this row's lane at o_taddr), where it still
// is, instead of reading back its partial: the same values, 1 / nk fewer
// bytes (called by whole warps then: the TMEM loads are warp-wide).
template <int D, bool OWN>
__device__ __forceinline__ void merge_rows(const float4* part, int nk, uint4* dst, int own,
                                           uint32_t o_taddr) {
  constexpr int NG = D / 4 + 1;
  const size_t piece_stride = static_cast<size_t>(2) * NG * BM;
  float m_all = -INFINITY;
  for (int k = 0; k < nk; ++k) m_all = fmaxf(m_all, __ldcg(part + k * piece_stride + (D / 4) * BM).x);
  float l_all = 0.f;
  for (int k = 0; k < nk; ++k) {
    const float4 ml = __ldcg(part + k * piece_stride + (D / 4) * BM);
    l_all = fmaf(ml.y, ex2(ml.x - m_all), l_all);
  }
  const float inv_l = 1.f / l_all;
  const uint64_t inv2 = pk2(inv_l, inv_l);
#pragma unroll
  for (int cg = 0; cg < D / 64; ++cg) {
    float acc[64];
#pragma unroll
    for (int e = 0; e < 64; ++e) acc[e] = 0.f;
    for (int k = 0; k < nk; ++k) {
      const float4* src = part + k * piece_stride;
      float4 v[16];
      if (OWN && k == own) {
        uint32_t t[64];
        tmem_ld32(o_taddr + cg * 64, t);
        tmem_ld32(o_taddr + cg * 64 + 32, t + 32);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e)
          v[e] = make_float4(__uint_as_float(t[4 * e]), __uint_as_float(t[4 * e + 1]),
                             __uint_as_float(t[4 * e + 2]), __uint_as_float(t[4 * e + 3]));
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = __ldcg(src + (cg * 16 + e) * BM);
      }
      const float a = ex2(__ldcg(src + (D / 4) * BM).x - m_all);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        acc[4 * e] = fmaf(v[e].x, a, acc[4 * e]);
        acc[4 * e + 1] = fmaf(v[e].y, a, acc[4 * e + 1]);
        acc[4 * e + 2] = fmaf(v[e].z, a, acc[4 * e + 2]);
        acc[4 * e + 3] = fmaf(v[e].w, a, acc[4 * e + 3]);
      }
    }
    if (dst) {
#pragma unroll
      for (int c = 0; c < 64; c += 8) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float o0, o1;
          up2(fmul2(pk2(acc[c + 2 * e], acc[c + 2 * e + 1]), inv2), o0, o1);
          w[e] = pack_bf16x2(o0, o1);
        }
        dst[(cg * 64 + c) / 8] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
}

// Counts one piece in on its arrival counter and returns how many pieces of
// this launch (epoch) were counted in before it, or -1 if the exchange kept
// failing (it cannot fail more often than there are pieces; the bound only
// guards the loop).  The counter holds (epoch << 32) | count; a value tagged
// with another epoch, left by an earlier launch that gave up, counts as 0.
__device__ __forceinline__ int count_in(unsigned long long* counter, unsigned int epoch) {
  unsigned long long cur = ld_relaxed_gpu(counter);
  for (int attempt = 0; attempt < 4 * MAX_PIECES + 64; ++attempt) {
    const unsigned int cnt =
        static_cast<unsigned int>(cur >> 32) == epoch ? static_cast<unsigned int>(cur) : 0u;
    const unsigned long long want = (static_cast<unsigned long long>(epoch) << 32) | (cnt + 1u);
    const unsigned long long prev = atom_cas_acq_rel_gpu(counter, cur, want);
    if (prev == cur) return static_cast<int>(cnt);
    cur = prev;
  }
  return -1;
}

// The merge, out of line so that its registers do not weigh on the softmax
// loop's allocation: every piece read back from the workspace ...
template <int D>
__device__ __noinline__ void merge_pieces(const float4* part, int nk, uint4* dst) {
  merge_rows<D, false>(part, nk, dst, -1, 0u);
}

// ... or, at D = 64, the merging piece's own O taken from TMEM.
template <int D>
__device__ __noinline__ void merge_pieces_own(const float4* part, int nk, uint4* dst, int own,
                                              uint32_t o_taddr) {
  merge_rows<D, true>(part, nk, dst, own, o_taddr);
}

// ----------------------------------------------------------------------------
// The kernel
// ----------------------------------------------------------------------------
// BC = false: dense and prefix-cached forms (every key visible).
// BC = true: block-causal form (one key segment, per-row image-id mask).
template <int D, bool BC>
// 10 or 11 warps on 4 SM sub-partitions (16 Ki registers each, 3 warps on
// two or three of them) cap a thread at 168 registers.
__global__ void __launch_bounds__(num_threads<D>(), 1)
    attn_fwd_kernel(const __grid_constant__ Params p) {
  using C = Cfg<D>;
  constexpr int NT = num_threads<D>();
  constexpr bool DUAL = C::P_OWN;  // two MMA warps, one per query tile
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle atoms.
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  SharedCtl* ctl = reinterpret_cast<SharedCtl*>(base + C::BAR_OFF);
  volatile int* abort_flag = &ctl->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T0 = p.n_tiles[0];
  const int T = T0 + p.n_tiles[1];
  const uint64_t limit = p.wait_limit_ns;

  const uint32_t ring = base_u32 + C::RING_OFF;
  const uint32_t qs = base_u32 + C::Q_OFF;
  const uint32_t bar_q = smem_u32(&ctl->q_full);
  const uint32_t bar_qfree = smem_u32(&ctl->q_free);
  auto bar_kv_full = [&](int s) { return smem_u32(&ctl->kv_full[s]); };
  auto bar_kv_empty = [&](int s) { return smem_u32(&ctl->kv_empty[s]); };
  // Per query tile (addresses computed, not indexed from an array: a runtime
  // index into a local array would put it in local memory).
  auto bar_s = [&](int i) { return smem_u32(&ctl->s_full[i]); };
  auto bar_p = [&](int i) { return smem_u32(&ctl->p_full[i]); };
  auto bar_o = [&](int i) { return smem_u32(&ctl->o_full[i]); };
  auto bar_ofree = [&](int i) { return smem_u32(&ctl->o_free[i]); };
  auto bar_ifull = [&](int s) { return smem_u32(&ctl->item_full[s]); };
  auto bar_iempty = [&](int s) { return smem_u32(&ctl->item_empty[s]); };
  Item* const item_ring = reinterpret_cast<Item*>(ctl->item_ring);
  auto bar_pvdone = [&](int i) { return smem_u32(&ctl->pv_done[i]); };
  auto bar_sfree = [&](int i) { return smem_u32(&ctl->s_free[i]); };

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    mbar_init(bar_qfree, DUAL ? 2 : 1);  // one release per MMA warp
    for (int s = 0; s < C::NRING; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), DUAL ? 2 : 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_s(i), 1);
      mbar_init(bar_p(i), 4);      // one arrival per softmax warp
      mbar_init(bar_o(i), 1);
      mbar_init(bar_ofree(i), 4);  // one arrival per softmax warp
      mbar_init(bar_pvdone(i), 1);
      mbar_init(bar_sfree(i), 4);  // one arrival per softmax warp
      mbar_init(smem_u32(&ctl->part_done[i]), 4);
      mbar_init(smem_u32(&ctl->merge_ready[i]), 1);
    }
    mbar_init(smem_u32(&ctl->drain), DUAL ? 2 : 1);
    mbar_init(smem_u32(&ctl->tail_ready), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_ifull(s), 1);
      mbar_init(bar_iempty(s), NT / 32 - 1);  // every warp but the loader
    }
    ctl->n_tail_items = MAX_CTA_TAIL_ITEMS;
    ctl->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == MMA_WARP) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ctl->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // Masked forms: summarise the image ids of every key tile (the roles' tile
  // walk needs it from their first item on).  Each warp takes 4 tiles at a
  // time with their loads in flight together; lane l summarises keys
  // 4 l .. 4 l + 3 of a tile, with one 16-byte load when the tile is whole and
  // 16-byte aligned (image_ids itself is).
  TileTable tt{nullptr};
  if constexpr (BC) {
    constexpr int NW = NT / 32;
    int* t_lo = reinterpret_cast<int*>(base + C::SUM_OFF);
    for (int t0 = warp; t0 < T; t0 += 4 * NW) {
      int id[4][4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int t = t0 + b * NW;
        if (t >= T) continue;
        const int pos0 = key_tile_pos(p, t), len = key_tile_len(p, t);
        if (len == BN && (pos0 & 3) == 0) {
          const int4 v = __ldg(reinterpret_cast<const int4*>(p.image_ids + pos0) + lane);
          id[b][0] = v.x;
          id[b][1] = v.y;
          id[b][2] = v.z;
          id[b][3] = v.w;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            id[b][e] = (4 * lane + e < len) ? __ldg(p.image_ids + pos0 + 4 * lane + e) : 0;
        }
      }
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int t = t0 + b * NW;
        if (t >= T) continue;  // warp-uniform
        const int len = key_tile_len(p, t);
        int lo = 0x7fffffff, hi = -1;
        bool text = false;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (4 * lane + e >= len) continue;  // past the tile's last key
          if (id[b][e] < 0) {
            text = true;
          } else {
            lo = min(lo, id[b][e]);
            hi = max(hi, id[b][e]);
          }
        }
        lo = __reduce_min_sync(0xffffffffu, lo);
        hi = __reduce_max_sync(0xffffffffu, hi);
        text = __any_sync(0xffffffffu, text);
        if (lane == 0) {
          t_lo[t] = lo;
          t_lo[MAX_SEQ_TILES + t] = hi;
          t_lo[2 * MAX_SEQ_TILES + t] = (!text && lo == hi) ? 1 : 0;
        }
      }
    }
    tt = TileTable{t_lo};
    // The unit order (see UnitOrder): visited tiles per query pair, then
    // each pair's rank, then the levels.
    int* ob = reinterpret_cast<int*>(base + C::ORDER_OFF);
    int* cnt = ob + ORDER_QP + MAX_Q_PAIRS;
    const int qpn = p.sc.q_pairs;
    for (int q = threadIdx.x; q < qpn; q += NT) cnt[q] = 0;
    __syncthreads();
    for (int x = threadIdx.x; x < qpn * T; x += NT) {
      const int q = x / T, t = x - q * T;
      Unit uq;
      uq.b = 0;
      uq.h = 0;
      uq.q0 = q * 2 * BM;
      uq.two = uq.q0 + BM < p.Nq;
      const int cost = bc_pair_tile_cost(tt, p, uq, t);
      if (cost) atomicAdd(&cnt[q], cost);
    }
    __syncthreads();
    for (int q = threadIdx.x; q < qpn; q += NT) ob[ORDER_QP + order_rank(cnt, qpn, q)] = q;
    __syncthreads();
    if (threadIdx.x == 0) order_levels(ob, cnt, qpn);
  }
  const bool masked_tail = BC && p.sc.tail_ctas > 0;
  const int* tail_pre = masked_tail ? reinterpret_cast<const int*>(base + C::TAIL_OFF) : nullptr;
  MaskedTail mtail{&p, tt, tail_pre, reinterpret_cast<const Item*>(base + C::ITEMS_OFF), 0,
                   UnitOrder{BC ? reinterpret_cast<const int*>(base + C::ORDER_OFF) : nullptr}};
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  // Masked forms with a split tail: the loader, which decodes every work item
  // for the other roles, waits before its first tail item until the softmax
  // warps have worked the tail items out.
  const int tail_rounds = p.sc.tail_ctas ? p.sc.n_whole / static_cast<int>(gridDim.x) : 0;
  const uint32_t bar_tail = smem_u32(&ctl->tail_ready);
  // (Called by the loader, whole warp.)
  auto await_tail = [&](int n, int site) -> bool {
    if (!masked_tail || n < tail_rounds || mtail.n_items > 0) return true;
    if (!warp_wait(bar_tail, 0, limit, abort_flag, site)) return false;
    mtail.n_items = ctl->n_tail_items;
    return true;
  };
  // Work item n, decoded once by the loader and read by the other roles
  // (whole warps).  The loader writes item n into slot n & 1 once every
  // reader is done with item n - 2 (item_empty), then arrives on item_full;
  // a slot with t_begin < 0 means no item is left.  A reader keeps the slot
  // of its current item (masked forms: its tile masks, below) until it takes
  // the next one.  take_item returns false at the end or, with ok false, when
  // a wait gave up.
  //
  // Masked forms: with each item the loader leaves three bit masks over the
  // key tiles [t_begin, t_end) in its slot (MASK_OFF): visited by the item's
  // query pair, and seen whole by query tile 0, by query tile 1.  The roles
  // test a bit per key tile instead of the tile tables.
  uint32_t* const tile_masks = reinterpret_cast<uint32_t*>(base + C::MASK_OFF);
  auto slot_masks = [&](int n) -> const uint32_t* {
    return tile_masks + (n & 1) * 3 * C::MASK_WORDS;
  };
  auto tile_bit = [](const uint32_t* m, int t) -> bool { return (m[t >> 5] >> (t & 31)) & 1u; };
  auto publish_item = [&](int n, const Item* src) -> bool {
    const int sl = n & 1;
    if (n >= 2 && !warp_wait(bar_iempty(sl), ((n >> 1) - 1) & 1, limit, abort_flag, 17))
      return false;
    if constexpr (BC) {
      if (src) {
        uint32_t* mk = tile_masks + sl * 3 * C::MASK_WORDS;
        const Unit& u = src->u;
        const int qt0 = u.q0 / BM;
        for (int w = src->t_begin >> 5; w <= (src->t_end - 1) >> 5; ++w) {
          const int t = w * 32 + lane;
          const bool vis = t >= src->t_begin && t < src->t_end && bc_unit_visits(tt, p, u, t);
          const bool f0 = vis && bc_tile_full(tt, p, qt0, u.q0, t);
          const bool f1 = vis && u.two && bc_tile_full(tt, p, qt0 + 1, u.q0 + BM, t);
          const uint32_t bv = __ballot_sync(0xffffffffu, vis);
          const uint32_t b0 = __ballot_sync(0xffffffffu, f0);
          const uint32_t b1 = __ballot_sync(0xffffffffu, f1);
          if (lane == 0) {
            mk[w] = bv;
            mk[C::MASK_WORDS + w] = b0;
            mk[2 * C::MASK_WORDS + w] = b1;
          }
        }
      }
    }
    if (lane == 0) {
      if (src) item_ring[sl] = *src; else item_ring[sl].t_begin = -1;
      mbar_arrive(bar_ifull(sl));
    }
    __syncwarp();
    return true;
  };
  auto take_item = [&](int n, Item& out, bool& ok) -> bool {
    const int sl = n & 1;
    if (n >= 1 && lane == 0) mbar_arrive(bar_iempty(sl ^ 1));  // done with item n - 1
    ok = warp_wait(bar_ifull(sl), (n >> 1) & 1, limit, abort_flag, 16);
    if (!ok) return false;
    out = item_ring[sl];
    __syncwarp();
    return out.t_begin >= 0;
  };
  // Loader bookkeeping for draining copies in flight after an abort.
  uint32_t ld_issued = 0, ld_parity = 0;  // per ring entry: a load was issued / its phase
  int q_last = -1;                        // last unit whose Q load was issued

  if (warp == PRODUCER_WARP) {
    // ---------------------------------------------------------------- loader
    // The whole warp runs the loop, converged; one elected lane issues each
    // copy (see mma_ss_elect).
    if (lane == 0) {
      prefetch_tmap(&p.tm_q);
      for (int s = 0; s < 2; ++s) {
        prefetch_tmap(&p.tm_k[s]);
        prefetch_tmap(&p.tm_v[s]);
      }
    }
    __syncwarp();
    {
      int slot = 0;
      uint32_t phase = 0;
      bool ok = true;
      Item it;
      for (int n = 0; ok; ++n) {
        ok = await_tail(n, 12);
        if (!ok) break;
        const bool has = get_item<BC>(p, &mtail, T, n, it);
        // Short units (prefetch_q): the next Q, read once from HBM, is
        // prefetched into L2 while the current item's last key tiles run.
        // Compiled into the dense D = 128 kernel only: present but unused, it
        // slowed the D = 64 one by ~2 % through code generation.
        if constexpr (!BC && D == 128) {
          if (p.sc.prefetch_q && has && n > 0) {
#pragma unroll
            for (int c = 0; c < C::CHUNKS; ++c) {
              tma_prefetch_4d_elect(&p.tm_q, c * 64, it.u.h, it.u.q0, it.u.b);
              if (it.u.two) tma_prefetch_4d_elect(&p.tm_q, c * 64, it.u.h, it.u.q0 + BM, it.u.b);
            }
          }
        }
        ok = publish_item(n, has ? &it : nullptr);
        if (!ok || !has) break;
        const Unit& u = it.u;
        // The Q buffers are free once every S MMA of the previous item is done.
        if (n > 0) {
          ok = warp_wait(bar_qfree, (n - 1) & 1, limit, abort_flag, 9);
          if (!ok) break;
        }
        const int nq_tiles = u.two ? 2 : 1;
        mbar_expect_tx_elect(bar_q, nq_tiles * C::TILE_BYTES);
        for (int i = 0; i < nq_tiles; ++i)
          for (int c = 0; c < C::CHUNKS; ++c)
            tma_load_4d_elect(qs + i * C::TILE_BYTES + c * C::CHUNK_BYTES, &p.tm_q, c * 64, u.h,
                              u.q0 + i * BM, u.b, bar_q);
        q_last = n;
        int prev_t = -1;  // D = 128: the last key tile of this item loaded so far
#pragma unroll 1
        for (int t = it.t_begin; t < it.t_end && ok; ++t) {
          if (BC && !tile_bit(slot_masks(n), t)) continue;
          const int seg = (t < T0) ? 0 : 1;
          const int tok0 = (t - (seg ? T0 : 0)) * BN;
          if constexpr (C::KV_PAIRS) {
            ok = warp_wait(bar_kv_empty(slot), phase ^ 1u, limit, abort_flag, 1);
            if (!ok) break;
            mbar_expect_tx_elect(bar_kv_full(slot), 2 * C::TILE_BYTES);
            for (int kind = 0; kind < 2; ++kind) {
              const bool skip = (p.fault_mode == 1) && kind == 1 && t == 1 && n == 0 && blockIdx.x == 0;
              if (skip) continue;
              const CUtensorMap* map = kind == 0 ? &p.tm_k[seg] : &p.tm_v[seg];
              for (int c = 0; c < C::CHUNKS; ++c)
                tma_load_4d_elect(ring + slot * C::ENTRY_BYTES + kind * C::TILE_BYTES +
                                      c * C::CHUNK_BYTES,
                                  map, c * 64, u.h, tok0, u.b, bar_kv_full(slot));
            }
            ld_issued |= 1u << slot;
            ld_parity = (ld_parity & ~(1u << slot)) | (phase << slot);
            if (++slot == C::NRING) {
              slot = 0;
              phase ^= 1u;
            }
          } else {
            ok = warp_wait(bar_kv_empty(slot), phase ^ 1u, limit, abort_flag, 1);
            if (!ok) break;
            mbar_expect_tx_elect(bar_kv_full(slot), (prev_t >= 0 ? 2 : 1) * C::TILE_BYTES);
            if (prev_t >= 0) {
              const bool skip = (p.fault_mode == 1) && prev_t == 1 && n == 0 && blockIdx.x == 0;
              const int vseg = (prev_t < T0) ? 0 : 1;
              const int vtok0 = (prev_t - (vseg ? T0 : 0)) * BN;
              if (!skip)
                for (int c = 0; c < C::CHUNKS; ++c)
                  tma_load_4d_elect(
                      ring + slot * C::ENTRY_BYTES + C::TILE_BYTES + c * C::CHUNK_BYTES,
                      &p.tm_v[vseg], c * 64, u.h, vtok0, u.b, bar_kv_full(slot));
            }
            for (int c = 0; c < C::CHUNKS; ++c)
              tma_load_4d_elect(ring + slot * C::ENTRY_BYTES + c * C::CHUNK_BYTES, &p.tm_k[seg],
                                c * 64, u.h, tok0, u.b, bar_kv_full(slot));
            ld_issued |= 1u << slot;
            ld_parity = (ld_parity & ~(1u << slot)) | (phase << slot);
            if (++slot == C::NRING) {
              slot = 0;
              phase ^= 1u;
            }
            prev_t = t;
          }
        }
        // D = 128: the item's last V, in an entry of its own.
        if (!C::KV_PAIRS && ok && prev_t >= 0) {
          ok = warp_wait(bar_kv_empty(slot), phase ^ 1u, limit, abort_flag, 1);
          if (!ok) break;
          mbar_expect_tx_elect(bar_kv_full(slot), C::TILE_BYTES);
          const bool skip = (p.fault_mode == 1) && prev_t == 1 && n == 0 && blockIdx.x == 0;
          const int vseg = (prev_t < T0) ? 0 : 1;
          const int vtok0 = (prev_t - (vseg ? T0 : 0)) * BN;
          if (!skip)
            for (int c = 0; c < C::CHUNKS; ++c)
              tma_load_4d_elect(ring + slot * C::ENTRY_BYTES + C::TILE_BYTES + c * C::CHUNK_BYTES,
                                &p.tm_v[vseg], c * 64, u.h, vtok0, u.b, bar_kv_full(slot));
          ld_issued |= 1u << slot;
          ld_parity = (ld_parity & ~(1u << slot)) | (phase << slot);
          if (++slot == C::NRING) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == MMA_WARP || (DUAL && warp == MMA_WARP2)) {
    // ----------------------------------------------------------- MMA issuers
    // The whole warp runs the loop, converged (warp-wide bounded waits); one
    // elected lane issues each MMA and commit (see mma_ss_elect).
    {
      constexpr uint32_t IDESC_S = make_idesc(BM, BN, false);
      constexpr uint32_t IDESC_PV = make_idesc(BM, D, true);
      // S_i = Q_i K^T over D in K-steps of 16 (32 bytes inside a 128-byte row).
      // The dense D = 128 kernel builds its descriptors once per group:
      // shared-memory addresses stay below 2^18, so the start-address field
      // (address / 16, 14 bits) of base + off is the base's plus off / 16,
      // with no carry out of it.  Measured, this suits only that kernel (the
      // D = 64 and masked ones were slower with it), so the others build each
      // MMA's descriptors from its address.
      constexpr bool BASE_DESC = (D == 128) && !BC;
      auto issue_s = [&](int i, uint32_t kb) {
        const uint32_t qa = qs + i * C::TILE_BYTES;
        const uint64_t qd = sw128_desc(qa, 16, 1024);
        const uint64_t kd = sw128_desc(kb, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
          if constexpr (BASE_DESC)
            mma_ss_elect(tmem + C::s_col(i), qd + (off >> 4), kd + (off >> 4), IDESC_S, kk > 0);
          else
            mma_ss_elect(tmem + C::s_col(i), sw128_desc(qa + off, 16, 1024),
                         sw128_desc(kb + off, 16, 1024), IDESC_S, kk > 0);
        }
      };
      // O_i += P_i V over the BN keys in K-steps of 16 rows of V (MN-major B).
      auto issue_pv = [&](int i, uint32_t vb, bool accumulate) {
        const uint64_t vd = sw128_desc(vb, C::CHUNK_BYTES, 1024);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts_elect(tmem + C::o_col(i), tmem + C::p_col(i) + kk * 8,
                       BASE_DESC ? vd + kk * (16 * 128 >> 4)
                                 : sw128_desc(vb + kk * 16 * 128, C::CHUNK_BYTES, 1024),
                       IDESC_PV, (accumulate || kk > 0) ? 1u : 0u);
      };

      if constexpr (C::P_OWN) {
        // D = 64, P in columns of its own; one MMA warp per query tile i.
        // Per visited key tile j: once the softmax warps have read S_i(j - 1)
        // (s_free), S_i(j) goes, and runs while they work on S_i(j - 1); then,
        // once P_i(j - 1) is written, P_i V(j - 1), which commits pv_done (the
        // softmax warps wait for it before writing P_i again or rescaling O_i);
        // an item's last P V commits o_full.  The K and V of a key tile share
        // one ring entry (KV_PAIRS), loaded in key-tile order; ld counts the
        // entries consumed.  Entry j - 1 is released after P_i V(j - 1), its
        // last reader.  A ring entry and the Q buffers are free once both
        // warps have released them (kv_empty and q_free take two arrivals): by
        // a commit after their MMAs, or, for an item without this warp's query
        // tile, by a plain arrival made after the entry's or Q's full phase, so
        // that it never counts toward the phase before.
        const int i = warp - MMA_WARP;  // this warp's query tile
        uint32_t si = 0;  // S issued (phases of s_full / p_full)
        uint32_t oc = 0;  // items finished (phases of o_full / o_free)
        uint32_t ld = 0;  // ring entries (key tiles, K and V together) consumed
        bool ok = true;
        auto ring_wait = [&](uint32_t x, int site) -> int {
          const int sl = static_cast<int>(x % C::NRING);
          if (!warp_wait(bar_kv_full(sl), (x / C::NRING) & 1u, limit, abort_flag, site)) return -1;
          return sl;
        };
        auto release = [&](uint32_t bar, bool mine) {
          if (mine) {
            mma_commit_elect(bar);
          } else {
            if (lane == 0) mbar_arrive(bar);
            __syncwarp();
          }
        };
        // P_i V(j - 1): P_i(j - 1) was waited for; the first of an item waits
        // for the epilogue that read O_i.
        auto pv = [&](uint32_t vb, bool accumulate) -> bool {
          if (!accumulate && oc > 0 &&
              !warp_wait(bar_ofree(i), (oc - 1u) & 1u, limit, abort_flag, 6))
            return false;
          tc_fence_after();
          issue_pv(i, vb, accumulate);
          return true;
        };
        Item it;
        for (int n = 0; ok && take_item(n, it, ok); ++n) {
          const bool mine = i == 0 || it.u.two;
          ok = warp_wait(bar_q, n & 1, limit, abort_flag, 2);
          if (!ok) break;
          int j = 0;      // key tiles visited so far in this item
          int prev = 0;   // ring entry of key tile j - 1
#pragma unroll 1
          for (int t = it.t_begin; t < it.t_end && ok; ++t) {
            if (BC && !tile_bit(slot_masks(n), t)) continue;
            const int e = ring_wait(ld, 3);
            ok = e >= 0;
            if (!ok) break;
            tc_fence_after();
            if (mine) {
              // S_i(j) overwrites S_i(j - 1): wait until the softmax warps
              // have read it (S number si - 1).  An item's first S follows
              // the previous item's last P, which they wrote after reading.
              if (j > 0) {
                ok = warp_wait(bar_sfree(i), (si - 1u) & 1u, limit, abort_flag, 18);
                if (!ok) break;
                tc_fence_after();
              }
              issue_s(i, ring + e * C::ENTRY_BYTES);
              mma_commit_elect(bar_s(i));
              ++si;
              if (j > 0) {
                // P_i(j - 1) is P number si - 2 (S_i(j) is counted already).
                ok = warp_wait(bar_p(i), (si - 2u) & 1u, limit, abort_flag, 4);
                if (!ok) break;
                tc_fence_after();
                ok = pv(ring + prev * C::ENTRY_BYTES + C::TILE_BYTES, j - 1 > 0);
                if (!ok) break;
                mma_commit_elect(bar_pvdone(i));
              }
            }
            // Key tile j - 1's entry: its S and its P V have been issued.
            if (j > 0) release(bar_kv_empty(prev), mine);
            prev = e;
            ++ld;
            ++j;
          }
          if (!ok) break;
          release(bar_qfree, mine);  // every S MMA of this item has been issued
          if (mine) {
            ok = warp_wait(bar_p(i), (si - 1u) & 1u, limit, abort_flag, 4);
            if (!ok) break;
            ok = pv(ring + prev * C::ENTRY_BYTES + C::TILE_BYTES, j - 1 > 0);
            if (!ok) break;
            mma_commit_elect(bar_o(i));
            ++oc;
          }
          release(bar_kv_empty(prev), mine);
        }
      } else {
      uint32_t ld = 0;            // ring entries consumed
      uint32_t sc[2] = {0u, 0u};  // S commits per query tile (phases of s_full / p_full)
      uint32_t oc[2] = {0u, 0u};  // units finished per query tile (phases of o_full / o_free)
      bool ok = true;
      auto ring_wait = [&](int site) -> int {
        const int sl = static_cast<int>(ld % C::NRING);
        if (!warp_wait(bar_kv_full(sl), (ld / C::NRING) & 1u, limit, abort_flag, site)) return -1;
        ++ld;
        return sl;
      };
      // The first P V of a unit overwrites O_i: wait until the epilogue of the
      // previous unit has read it out of TMEM.
      auto pv = [&](int i, uint32_t vb, bool accumulate) -> bool {
        if (!warp_wait(bar_p(i), (sc[i] - 1u) & 1u, limit, abort_flag, 4)) return false;
        if (!accumulate && oc[i] > 0 &&
            !warp_wait(bar_ofree(i), (oc[i] - 1u) & 1u, limit, abort_flag, 6))
          return false;
        tc_fence_after();
        issue_pv(i, vb, accumulate);
        return true;
      };
      Item it;
      for (int n = 0; ok && take_item(n, it, ok); ++n) {
        const int nq = it.u.two ? 2 : 1;
        ok = warp_wait(bar_q, n & 1, limit, abort_flag, 2);
        if (!ok) break;
        int j = 0;  // key tiles visited so far in this item
#pragma unroll 1
        for (int t = it.t_begin; t < it.t_end && ok; ++t) {
          if (BC && !tile_bit(slot_masks(n), t)) continue;
          // Entry of key tile j: K_j, and V_{j-1} when j > 0.
          const int e = ring_wait(3);
          ok = e >= 0;
          if (!ok) break;
          tc_fence_after();
          const uint32_t kb = ring + e * C::ENTRY_BYTES;
          // Unrolled over the two query tiles, so that sc[] / oc[] are
          // indexed by constants and stay in registers.
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (i >= nq || !ok) break;
            if (j > 0) {
              ok = pv(i, kb + C::TILE_BYTES, j - 1 > 0);
              if (!ok) break;
            }
            issue_s(i, kb);
            mma_commit_elect(bar_s(i));
            ++sc[i];
          }
          if (!ok) break;
          mma_commit_elect(bar_kv_empty(e));
          ++j;
        }
        if (!ok) break;
        mma_commit_elect(bar_qfree);  // every S MMA of this item has been issued
        // The entry after the last key tile: the last V alone.
        const int e = ring_wait(5);
        ok = e >= 0;
        if (!ok) break;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (i >= nq || !ok) break;
          ok = pv(i, ring + e * C::ENTRY_BYTES + C::TILE_BYTES, j - 1 > 0);
          if (!ok) break;
          mma_commit_elect(bar_o(i));
          ++oc[i];
        }
        if (ok) mma_commit_elect(bar_kv_empty(e));
      }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------- softmax / correction / store
    const int i = warp >> 2;  // query tile
    const int wq = warp & 3;  // TMEM lane quarter
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + C::s_col(i);
    const uint32_t p_addr = tmem + lane_base + C::p_col(i);
    const uint32_t o_addr = tmem + lane_base + C::o_col(i);
    const float sl2 = p.scale_log2;
    uint32_t sc = 0, oc = 0;  // phases of s_full / p_full and of o_full / o_free
    uint32_t pvc = 0;         // D = 64: phases of pv_done waited
    bool ok = true;
    uint32_t mc = 0;  // split items done by this query tile (phases of part_done / merge_ready)
    const uint32_t bar_part = smem_u32(&ctl->part_done[i]);
    const uint32_t bar_merge = smem_u32(&ctl->merge_ready[i]);
    const int row = wq * 32 + lane;  // row of the 128-row query tile (= TMEM lane)
    if (masked_tail) {
      // The split tail's schedule, worked out by the 8 softmax warps (named
      // barrier 1, before any bounded wait of theirs) while the loader and the
      // MMA issuer start on the whole units: the visited tiles of each tail
      // unit (one (unit, tile) pair per thread, shared-memory atomics), their
      // prefix sums (warp 0, shuffles), then this CTA's tail items, warp w
      // taking items w, w + 8, ... (ballots over a unit's key tiles find its
      // v-th visited tile).  Item j exists iff items 0 .. j - 1 do, so the
      // count is the first missing one.
      constexpr int NS = 8 * 32;
      int* pre = reinterpret_cast<int*>(base + C::TAIL_OFF);
      const int n_tail = p.sc.tail_units;
      for (int r = threadIdx.x; r <= n_tail; r += NS) pre[r] = 0;
      named_barrier(1, NS);
      for (int x = threadIdx.x; x < n_tail * T; x += NS) {
        const int r = x / T, t = x - r * T;
        if (bc_unit_visits(tt, p, decode_unit(p.sc, true, p.sc.n_whole + r, &mtail.ord), t))
          atomicAdd(&pre[r + 1], 1);
      }
      named_barrier(1, NS);
      if (warp == 0) {
        int carry = 0;
        for (int r0 = 0; r0 < n_tail; r0 += 32) {
          const int r = r0 + lane;
          int v = r < n_tail ? pre[r + 1] : 0;
#pragma unroll
          for (int d = 1; d < 32; d <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, v, d);
            if (lane >= d) v += x;
          }
          if (r < n_tail) pre[r + 1] = carry + v;
          carry += __shfl_sync(0xffffffffu, v, 31);
        }
      }
      named_barrier(1, NS);
      {
        Item* items = reinterpret_cast<Item*>(base + C::ITEMS_OFF);
        auto to_tile = [&](const Unit& uu, int v) {
          int seen = 0;
          for (int t0 = 0; t0 < T; t0 += 32) {
            const int t = t0 + lane;
            unsigned int msk = __ballot_sync(0xffffffffu, t < T && bc_unit_visits(tt, p, uu, t));
            const int cnt = __popc(msk);
            if (v < seen + cnt) {
              for (int skip = v - seen; skip > 0; --skip) msk &= msk - 1;  // drop lower set bits
              return t0 + __ffs(msk) - 1;
            }
            seen += cnt;
          }
          return T - 1;
        };
        const MaskedTail mt0{&p, tt, pre, nullptr, 0, mtail.ord};
        for (int jj = warp; jj < MAX_CTA_TAIL_ITEMS; jj += 8) {
          Item ti;
          if (masked_tail_item(p.sc, mt0, T, static_cast<int>(blockIdx.x), jj, ti, to_tile)) {
            if (lane == 0) items[jj] = ti;
          } else {
            if (lane == 0) atomicMin(&ctl->n_tail_items, jj);
            break;
          }
        }
      }
      named_barrier(1, NS);
      if (threadIdx.x == 0) mbar_arrive(bar_tail);
      mtail.n_items = ctl->n_tail_items;
    }
    Item it;
    for (int n = 0; ok && take_item(n, it, ok); ++n) {
      const Unit& u = it.u;
      if (i == 1 && !u.two) continue;
      float m = -INFINITY;  // running (possibly stale) maximum, log2 units
      float l = 0.f;        // running sum of exp2(x - m)
      RowMask mask{0, 0, -1, u.b, false, false};
      if constexpr (BC) {
        const int qrow = u.q0 + i * BM + row;  // query index; past Nq: a padding row
        mask.qi = p.n_tok[0] + qrow;
        mask.idq = qrow < p.Nq ? __ldg(p.image_ids + mask.qi) : -1;
      }
      int j = 0;  // key tiles visited so far in this item
#pragma unroll 1
      for (int t = it.t_begin; t < it.t_end; ++t) {
        if constexpr (BC) {
          const uint32_t* mk = slot_masks(n);
          if (!tile_bit(mk, t)) continue;
          const bool full = tile_bit(mk + (1 + i) * C::MASK_WORDS, t);
          mask.c0 = key_tile_pos(p, t);
          mask.ids = !full;
          mask.valid = p.key_valid != nullptr;
        }
        uint32_t vis[4] = {~0u, ~0u, ~0u, ~0u};
        bool masked = false;
        if constexpr (BC) build_row_mask(p, mask, vis, masked);
        ok = warp_wait(bar_s(i), sc & 1u, limit, abort_flag, 7);
        if (!ok) break;
        ++sc;
        tc_fence_after();
        // Keys past the end of this segment: TMA filled them with zeros, their
        // scores must be -inf instead.
        const int seg = (t < T0) ? 0 : 1;
        const int valid = p.n_tok[seg] - (t - (seg ? T0 : 0)) * BN;
        // D = 64: P_i and O_i may be written once the previous P V is complete
        // (an item's first tile: the previous item's last P V, which its
        // epilogue waited for).
        const bool first = j == 0;
        auto before_store = [&]() -> bool {
          if constexpr (C::P_OWN) {
            if (!first) {
              if (!warp_wait(bar_pvdone(i), pvc & 1u, limit, abort_flag, 15)) return false;
              ++pvc;
              tc_fence_after();
            }
          }
          return true;
        };
        // D = 64: S_i may be overwritten by the next S once these warps
        // have read it.
        auto after_read = [&]() {
          if constexpr (C::P_OWN) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_sfree(i));
          }
        };
        ok = softmax_tile<D, BC>(s_addr, p_addr, o_addr, valid, sl2, !first, vis, masked, m, l,
                                 after_read, before_store);
        ++j;
        if (!ok) break;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_p(i));
      }
      if (!ok) break;
      ok = warp_wait(bar_o(i), oc & 1u, limit, abort_flag, 8);
      if (!ok) break;
      ++oc;
      tc_fence_after();
      // Epilogue: read O_i out of TMEM and release it to the next item's P V.
      // At D = 64 a tail piece releases it only once the merge, which reads
      // it again, is done (the next item's first P V waits for these warps'
      // first P anyway); measured, this suits D = 64 and not D = 128.
      constexpr bool OWN_FROM_TMEM = (D == 64);
      uint32_t r[D];
#pragma unroll
      for (int c = 0; c < D; c += 32) tmem_ld32(o_addr + c, r + c);
      tmem_wait_ld();
      auto release_o = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_ofree(i));
      };
      if (!OWN_FROM_TMEM || it.tail < 0) release_o();

      const int q = u.q0 + i * BM + row;  // this thread's query row
      uint4* dst = reinterpret_cast<uint4*>(
          p.out + ((static_cast<size_t>(u.b) * p.Nq + q) * p.H + u.h) * D);
      if (it.tail >= 0) {
        // A piece of a tail unit: publish (O, m, l) of this row, count the
        // piece in; the last piece of the unit to arrive merges every piece.
        // A piece's partial for one query tile is D / 4 + 1 groups of four
        // floats per row, group-major (group g of row r at g * 128 + r; the
        // last group holds m and l), so a warp's access to one group is 512
        // contiguous bytes.
        constexpr int NG = D / 4 + 1;
        auto part = [&](int k) {
          return reinterpret_cast<float4*>(p.ws_part) +
                 (static_cast<size_t>(it.slot0 + k) * 2 + i) * NG * BM + row;
        };
        {
          float4* w = part(it.piece);
#pragma unroll
          for (int g = 0; g < D / 4; ++g)
            __stcg(w + g * BM, make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                                           __uint_as_float(r[4 * g + 2]),
                                           __uint_as_float(r[4 * g + 3])));
          __stcg(w + (D / 4) * BM, make_float4(m, l, 0.f, 0.f));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_part);
        // The first warp of the tile counts the piece in.  It waits as a whole
        // warp: a lane spinning on one barrier while another lane of the same
        // warp spins on a different one serialises the two, and the waits
        // then run up to the hardware's suspend limit in turn.
        if (wq == 0) {
          ok = warp_wait(bar_part, mc & 1u, limit, abort_flag, 10);
          if (ok && lane == 0) {
            // Release this tile's partial (the other warps' writes were
            // acquired through bar_part) and, if last, acquire every piece's.
            const int before = count_in(p.ws_count + it.tail * 2 + i, p.epoch);
            if (before < 0) {
              *abort_flag = 1;
              record_timeout(14);
            }
            ctl->last[i] = before == it.pieces - 1;
            mbar_arrive(bar_merge);
          }
          __syncwarp();
        }
        ok = warp_wait(bar_merge, mc & 1u, limit, abort_flag, 11);
        ++mc;
        if (!ok) break;
        const float4* part0 = reinterpret_cast<const float4*>(p.ws_part) +
                              static_cast<size_t>(it.slot0 * 2 + i) * (D / 4 + 1) * BM + row;
        if constexpr (OWN_FROM_TMEM) {
          if (*reinterpret_cast<volatile int*>(&ctl->last[i]))
            merge_pieces_own<D>(part0, it.pieces, q < p.Nq ? dst : nullptr, it.piece, o_addr);
          release_o();
        } else {
          if (!*reinterpret_cast<volatile int*>(&ctl->last[i])) continue;
          merge_pieces<D>(part0, it.pieces, q < p.Nq ? dst : nullptr);
        }
        continue;
      }

      // A whole unit: O / l -> bf16 -> this thread's output row, in 32-byte
      // stores when the output is 32-byte aligned (rows are D * 2 bytes apart),
      // else in 16-byte ones.  The rows of a warp are H * D * 2 bytes apart, so
      // every store of the warp writes 32 separate sectors; whole sectors
      // halve the write requests at the end of each work item.
      if (q < p.Nq) {
        const float inv_l = 1.f / l;
        const uint64_t inv2 = pk2(inv_l, inv_l);
        if ((reinterpret_cast<uintptr_t>(p.out) & 31u) == 0) {
#pragma unroll
          for (int c = 0; c < D; c += 16) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              float a0, a1;
              up2(fmul2(pk2(__uint_as_float(r[c + 2 * e]), __uint_as_float(r[c + 2 * e + 1])), inv2),
                  a0, a1);
              w[e] = pack_bf16x2(a0, a1);
            }
            st_global_v8(dst + c / 8, w);
          }
        } else {
#pragma unroll
          for (int c = 0; c < D; c += 8) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float a0, a1;
              up2(fmul2(pk2(__uint_as_float(r[c + 2 * e]), __uint_as_float(r[c + 2 * e + 1])), inv2),
                  a0, a1);
              w[e] = pack_bf16x2(a0, a1);
            }
            dst[c / 8] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // Some role gave up: before the CTA exits and TMEM is released, let every
    // TMA copy and every MMA still in flight land (bounded waits again).
    if (warp == PRODUCER_WARP && lane == 0) {
      if (q_last >= 0) wait_drain(bar_q, q_last & 1, limit);
      for (int s = 0; s < C::NRING; ++s)
        if (ld_issued & (1u << s)) wait_drain(bar_kv_full(s), (ld_parity >> s) & 1u, limit);
    }
    if (warp == MMA_WARP || (DUAL && warp == MMA_WARP2)) {
      // The MMAs were issued by the elected lane: commit from it too.
      mma_commit_elect(smem_u32(&ctl->drain));
      if (lane == 0) wait_drain(smem_u32(&ctl->drain), 0, limit);
    }
    __syncwarp();
  }
  if (warp == MMA_WARP) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// Test probe of the two exp2 paths the softmax uses: mode 0 the FMA-pipe
// polynomial, mode 1 the MUFU ex2.approx.  One thread per pair of elements.
__global__ void exp2_probe_kernel(const float* __restrict__ x, float* __restrict__ y, long long n,
                                  int mode) {
  const long long k = 2 * (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x);
  if (k >= n) return;
  const bool pair = k + 1 < n;
  const float a = x[k];
  const float b = pair ? x[k + 1] : 0.f;
  float y0, y1;
  if (mode == 0) {
    exp2_poly2(pk2(a, b), y0, y1);
  } else {
    y0 = ex2(a);
    y1 = ex2(b);
  }
  y[k] = y0;
  if (pair) y[k + 1] = y1;
}

}  // namespace ncp
