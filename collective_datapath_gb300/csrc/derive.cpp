// derive.cpp -- layout-to-schedule deriver (see derive.h).
#include "derive.h"

#include <algorithm>
#include <map>
#include <utility>

#include "../../include/coll.h"
#include "policy_table.h"

namespace coll {

int line_bytes(int enc) {
  return enc == ENC_LL8 ? kLL8LineBytes : (enc == ENC_SENT ? kSentLineBytes : kLL128LineBytes);
}
int line_elems(int enc) {
  return enc == ENC_LL8 ? kLL8Elems : (enc == ENC_SENT ? kSentElems : kLL128Elems);
}

uint64_t lines_for(int enc, uint64_t elems) {
  const uint64_t e = (uint64_t)line_elems(enc);
  return (elems + e - 1) / e;
}

// Partition rule: M = roundup(ceil(count / n), 8); partition r covers
// [r*M, min(count, (r+1)*M)).  Equal partitions whenever 8n divides count.
uint64_t shard_elems(uint64_t count, int n) {
  const uint64_t per = (count + (uint64_t)n - 1) / (uint64_t)n;
  return (per + 7) / 8 * 8;
}
uint64_t shard_begin(uint64_t count, int n, int r) {
  return std::min<uint64_t>(count, (uint64_t)r * shard_elems(count, n));
}
uint64_t shard_len(uint64_t count, int n, int r) {
  const uint64_t b = shard_begin(count, n, r);
  return std::min<uint64_t>(count, b + shard_elems(count, n)) - b;
}

static uint64_t round_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

// Segments in image order; each starts on a 4-line boundary (one LL8 group
// of a 16-byte chunk, one LL128 warp row).
static uint64_t build_image(int enc, const std::vector<std::pair<uint64_t, uint64_t>>& parts,
                            std::vector<Seg>& segs) {
  uint64_t line = 0;
  segs.clear();
  for (auto& pr : parts) {
    Seg s;
    s.line0 = line;
    s.elems = pr.first;
    s.in_elem = pr.second;
    s.lines = lines_for(enc, s.elems);
    segs.push_back(s);
    line += round_up(s.lines, 4);
  }
  return line;
}

namespace {

struct Tiler {
  uint64_t tile;  // lines per tile, a multiple of 4
  int enc;
  template <class F>
  void over(const Seg& s, F&& f) const {
    for (uint64_t t0 = 0; t0 < s.lines; t0 += tile) {
      const uint64_t nl = std::min<uint64_t>(tile, s.lines - t0);
      const uint64_t e0 = t0 * (uint64_t)line_elems(enc);
      const uint64_t ne = std::min<uint64_t>(s.elems - e0, nl * (uint64_t)line_elems(enc));
      f(t0, nl, ne);
    }
  }
};

struct Counters {
  std::map<std::pair<int, uint64_t>, uint32_t> keys;
  uint32_t get(int space, uint64_t key) {
    auto it = keys.find({space, key});
    if (it != keys.end()) return it->second;
    const uint32_t id = (uint32_t)keys.size();
    keys[{space, key}] = id;
    return id;
  }
};

Item make_item(uint8_t kind, uint8_t dst, uint8_t src, uint64_t src_line, uint64_t nl,
               uint64_t ne, uint64_t out_off) {
  Item it{};
  it.kind = kind;
  it.dst = dst;
  it.src = src;
  it.src_line = src_line;
  it.nlines = (uint32_t)nl;
  it.nelems = (uint32_t)ne;
  it.out_off = out_off;
  return it;
}

void set_reset(Item& it, int readers, uint32_t counter) {
  if (readers <= 1) {
    it.flags |= IF_RESET_SOLE;
  } else {
    it.flags |= IF_RESET_COUNTED;
    it.readers = (uint16_t)readers;
    it.counter = counter;
  }
}

// Group items by destination rank and fill the begin offsets.
void group_by_dst(std::vector<Item>& items, int n, int* beg) {
  std::stable_sort(items.begin(), items.end(),
                   [](const Item& a, const Item& b) { return a.dst < b.dst; });
  int k = 0;
  for (int r = 0; r <= n; ++r) {
    while (k < (int)items.size() && items[k].dst < r) ++k;
    beg[r] = k;
  }
  for (int r = n + 1; r <= kMaxRanks; ++r) beg[r] = (int)items.size();
}

}  // namespace

// MoE dispatch: no work lists (the routing is only known on the device);
// the plan fixes the staging geometry and the device tables.
static int derive_moe(const DeriveInput& in, Plan& p) {
  const int n = in.nranks;
  if (in.encoding != COLL_LL128 && in.encoding != COLL_ENC_AUTO) return COLL_ERR_UNSUPPORTED;
  if (in.tokens < 0 || in.hidden <= 0 || in.topk < 1 || in.topk > 64 || in.experts < n ||
      in.experts % n != 0 || in.experts > 1024 || in.max_rows < 0)
    return COLL_ERR_INVALID;
  if (in.hidden % 8 != 0) return COLL_ERR_ALIGN;
  if (in.hidden > 48 * 1024) return COLL_ERR_UNSUPPORTED;  // two rows in shared memory
  p.kind = CK_MOE;
  p.enc = ENC_LL128;
  p.n = n;
  p.algorithm = 0;
  // streamed: routing, stage, copy launches; composed: routing, then one
  // launch of stage and copy tasks (staged rows read from L2)
  if (in.path != COLL_PATH_AUTO && in.path != COLL_PATH_STREAMED && in.path != COLL_PATH_COMPOSED)
    return COLL_ERR_UNSUPPORTED;
  p.path = in.path == COLL_PATH_AUTO ? COLL_PATH_COMPOSED : in.path;
  p.reset_mode = COLL_RESET_NONE;
  p.timeout_ns = in.timeout_ns ? in.timeout_ns : 200000000ull;
  p.moe_tokens = in.tokens;
  p.moe_hidden = in.hidden;
  p.moe_k = in.topk;
  p.moe_experts = in.experts;
  p.moe_el = in.experts / n;
  p.moe_nblocks = (in.tokens + kMoeBlockTokens - 1) / kMoeBlockTokens;
  p.moe_row_lines = (uint32_t)round_up(lines_for(ENC_LL128, (uint64_t)in.hidden), 4);
  const uint64_t worst = (uint64_t)in.tokens * n * std::min(in.topk, p.moe_el);
  p.moe_max_rows = (uint32_t)(in.max_rows > 0 ? std::min<uint64_t>(in.max_rows, worst) : worst);
  for (int r = 0; r < n; ++r) {
    p.in_elems[r] = (uint64_t)in.tokens * in.hidden;
    p.out_elems[r] = (uint64_t)p.moe_max_rows * in.hidden;
  }
  for (int r = 0; r <= kMaxRanks; ++r) p.sbeg[r] = p.beg1[r] = p.beg2[r] = 0;
  p.ctas_per_rank = 1;
  p.consume_grid = 1;
  uint64_t off = round_up(sizeof(WsHeader), 256);
  p.off_sitems = p.off_items1 = p.off_items2 = off;
  auto table = [&](uint64_t bytes) {
    const uint64_t o = off;
    off = round_up(off + std::max<uint64_t>(bytes, 4), 256);
    return o;
  };
  const uint64_t tk = (uint64_t)in.tokens * in.topk;
  p.off_entry_rank = table(4 * n * tk);
  p.off_block_off = table(4ull * n * p.moe_nblocks * in.experts);
  p.off_cnt = table(4ull * n * in.experts);
  p.off_tok_rank = table(4ull * n * in.tokens * n);
  p.off_dblock_off = table(4ull * n * p.moe_nblocks * n);
  p.off_stage_off = table(4ull * n * n);
  p.off_out_off = table(4ull * n * p.moe_el * n);
  p.off_rows_dest = table(4ull * n);
  p.off_counts_out = table(4ull * (n * p.moe_el * n + n));
  p.off_moe_flags = table(8ull * n * p.moe_nblocks * kMoeSubs);
  p.off_counters = table(4);
  off = round_up(off, 4096);
  // one staged row per (token, destination holding one of its experts)
  p.p_rank_lines = (uint64_t)in.tokens * std::min(in.topk, n) * p.moe_row_lines;
  p.P.rank_bytes = round_up(p.p_rank_lines * kLL128LineBytes, 4096);
  p.P.slot_bytes = p.P.rank_bytes * (uint64_t)n;
  p.P.slot_mask = (uint64_t)p.slots - 1;
  p.P.base = off;
  off += (uint64_t)p.slots * p.P.slot_bytes;
  p.ws_bytes = off;
  return COLL_OK;
}

// The calibrated entry for `n` ranks and `bytes` per rank: the table of the
// smallest calibrated group of at least n ranks (the largest one past it).
static const PolicyEntry* policy_lookup(int n, uint64_t bytes) {
  int group = kPolicyGroups[sizeof(kPolicyGroups) / sizeof(int) - 1];
  for (int g : kPolicyGroups)
    if (g >= n) {
      group = g;
      break;
    }
  int len = 0;
  const PolicyEntry* t = policy_table(group, &len);
  for (int i = 0; i < len; ++i)
    if (bytes <= t[i].max_bytes) return &t[i];
  return &t[len - 1];
}

int derive(const DeriveInput& in, Plan& p) {
  p = Plan{};
  const int n = in.nranks;
  // flash-comm §4.2: slots rotate with a device-side call counter; two
  // suffice here (a run starts after the previous one ended), four delay a
  // slot's reuse by three more runs
  if (in.slots != 0 && in.slots != 2 && in.slots != 4) return COLL_ERR_INVALID;
  p.slots = in.slots == 0 ? 2 : in.slots;
  if (n < 1 || n > kMaxRanks) return COLL_ERR_UNSUPPORTED;
  if (in.dtype != COLL_BF16 && in.dtype != COLL_F32) return COLL_ERR_UNSUPPORTED;
  // Sizes below are kept in 16-bit units: an fp32 element is two of them.
  // Counts and partitions are given and cut in elements of the dtype.
  const uint64_t eu = in.dtype == COLL_F32 ? 2 : 1;
  p.dtype = in.dtype;
  if (in.encoding != COLL_LL8 && in.encoding != COLL_LL128 && in.encoding != COLL_SENT &&
      in.encoding != COLL_ENC_AUTO)
    return COLL_ERR_UNSUPPORTED;
  if (in.reset_mode < 0 || in.reset_mode > 3 || in.path < 0 || in.path > 3 ||
      in.algorithm < 0 || in.algorithm > 2 || in.ctas < 0 || in.tile_lines < 0)
    return COLL_ERR_INVALID;

  const int L = in.in_layout, O = in.out_layout;
  if (L == COLL_SCATTERED && O == COLL_SCATTERED && in.op == COLL_REDUCE)
    p.kind = CK_ALLREDUCE;
  else if (L == COLL_SCATTERED && O == COLL_PACKED && in.op == COLL_REDUCE)
    p.kind = CK_REDUCE_SCATTER;
  else if (L == COLL_PACKED && O == COLL_SCATTERED && in.op == COLL_COPY)
    p.kind = CK_ALLGATHER;
  else if (L == COLL_SCATTERED && O == COLL_TRANSPOSED && in.op == COLL_COPY)
    p.kind = CK_ALLTOALL;
  else if (L == COLL_SCATTERED_V && O == COLL_PACKED_V && in.op == COLL_REDUCE)
    p.kind = CK_REDUCE_SCATTER_V;
  else if (L == COLL_PACKED_V && O == COLL_SCATTERED_V && in.op == COLL_COPY)
    p.kind = CK_ALLGATHER_V;
  else if (L == COLL_SCATTERED_V && O == COLL_TRANSPOSED_V && in.op == COLL_COPY) {
    if (in.experts > 0) {
      // a dispatch copies rows: an fp32 row is 2 * hidden 16-bit units, and
      // the plan's element counts are those units (coll_buffer_elems
      // divides them back)
      if (in.hidden % 8 != 0) return COLL_ERR_ALIGN;
      DeriveInput m = in;
      m.hidden = in.hidden * (int)eu;
      return derive_moe(m, p);
    }
    p.kind = CK_ALLTOALL_V;
  } else
    return COLL_ERR_UNSUPPORTED;

  // V collectives: runtime sizes (Purlin §3.1, V layouts), each a multiple
  // of 8 elements so that every segment starts 16-byte aligned.
  const bool vkind = p.kind == CK_REDUCE_SCATTER_V || p.kind == CK_ALLGATHER_V ||
                     p.kind == CK_ALLTOALL_V;
  std::vector<uint64_t> V;  // [n] or [n * n]
  uint64_t count_in = in.count;
  if (vkind) {
    const size_t want = p.kind == CK_ALLTOALL_V ? (size_t)n * n : (size_t)n;
    if (in.vcounts.size() != want) return COLL_ERR_INVALID;
    V = in.vcounts;
    uint64_t sum = 0;
    for (uint64_t v : V) {
      if (v % 8 != 0) return COLL_ERR_ALIGN;
      if (v > (1ull << 40)) return COLL_ERR_INVALID;
      sum += v;
    }
    if (p.kind != CK_ALLTOALL_V && sum != in.count) return COLL_ERR_INVALID;
    if (p.kind == CK_ALLTOALL_V) count_in = 0;
    for (uint64_t& v : V) v *= eu;
  }

  if (count_in % 8 != 0) return COLL_ERR_ALIGN;
  p.n = n;
  p.count = count_in * eu;
  p.shard = shard_elems(count_in, n) * eu;
  p.timeout_ns = in.timeout_ns ? in.timeout_ns : 200000000ull;
  if (p.kind == CK_ALLTOALL && shard_elems(count_in, n) * (uint64_t)n != in.count)
    return COLL_ERR_ALIGN;  // the exchange needs equal partitions

  const uint64_t count = p.count, M = p.shard;
  // partition k of the (elementwise) partition rule, in 16-bit units
  auto SB = [&](int k) { return shard_begin(count_in, n, k) * eu; };
  auto SL = [&](int k) { return shard_len(count_in, n, k) * eu; };
  uint64_t in_bytes_per_rank = 0;
  for (int r = 0; r < n; ++r) {
    switch (p.kind) {
      case CK_ALLREDUCE: p.in_elems[r] = count; p.out_elems[r] = count; break;
      case CK_REDUCE_SCATTER: p.in_elems[r] = count; p.out_elems[r] = SL(r); break;
      case CK_ALLGATHER: p.in_elems[r] = SL(r); p.out_elems[r] = count; break;
      case CK_ALLTOALL: p.in_elems[r] = count; p.out_elems[r] = count; break;
      case CK_REDUCE_SCATTER_V: p.in_elems[r] = count; p.out_elems[r] = V[r]; break;
      case CK_ALLGATHER_V: p.in_elems[r] = V[r]; p.out_elems[r] = count; break;
      case CK_ALLTOALL_V:
        p.in_elems[r] = p.out_elems[r] = 0;
        for (int k = 0; k < n; ++k) {
          p.in_elems[r] += V[(size_t)r * n + k];
          p.out_elems[r] += V[(size_t)k * n + r];
        }
        break;
      default: break;
    }
    in_bytes_per_rank = std::max<uint64_t>(in_bytes_per_rank, 2 * p.in_elems[r]);
  }

  // Encoding, algorithm and path.  An all-reduce with all three on AUTO
  // takes the calibrated policy entry for its group and size (flash-comm
  // §3.2 and §4.1: a constant-time lookup in a table measured offline).
  int enc = in.encoding, algo = in.algorithm, path = in.path;
  int ctas = in.ctas;  // the launch shape: 0 = the default width
  if (p.kind == CK_ALLREDUCE && enc == COLL_ENC_AUTO && algo == COLL_ALGO_AUTO &&
      path == COLL_PATH_AUTO) {
    const PolicyEntry* e = policy_lookup(n, in_bytes_per_rank);
    enc = e->enc;
    algo = e->algo;
    path = e->path;
    if (ctas == 0) ctas = e->ctas;
  }
  // Otherwise an AUTO encoding halves the bytes of small messages with
  // sentinel packs and uses LL128 lines above 1 MiB per rank.
  if (enc == COLL_ENC_AUTO) enc = in_bytes_per_rank <= (1u << 20) ? COLL_SENT : COLL_LL128;
  // Sentinel packs carry no epoch: without a re-arm a consumed pack would
  // look published to the next run of its slot.
  if (enc == COLL_SENT && in.reset_mode == COLL_RESET_NONE) {
    if (in.encoding == COLL_SENT) return COLL_ERR_UNSUPPORTED;
    enc = COLL_LL8;
  }
  p.enc = enc;
  p.reset_mode = p.enc == ENC_LL128 ? COLL_RESET_NONE : in.reset_mode;

  // Algorithm and path left on AUTO: boundaries placed on measured points
  // of the 8-rank sweeps on GB300.  Oneshot up to 512 KiB per rank (it reads
  // N^2 S of lines but has one phase), twoshot above; one fused cooperative
  // kernel up to 256 KiB per rank for LL8 and sentinel packs; the composed
  // launch for the LL128 twoshot and reduce-scatter (8 x 1 MiB reduce-
  // scatter: 18 against 40 us stream-ordered), for the LL128 all-gather
  // (equal up to 16 MiB, then faster: 8 x 256 MiB 0.40 against 0.55 ms) and
  // for the all-to-all from 4 MiB (8 x 4 MiB: 32 against 34 us); the V forms
  // follow the same rules (Zipf split of 256 MiB: reduce-scatter V 0.58
  // against 1.11 ms, all-gather V 0.40 against 0.55, all-to-all V 0.87
  // against 1.44); stream-
  // ordered kernels otherwise.  Two ranks always use oneshot (both move S
  // per rank).
  p.algorithm = 0;
  if (p.kind == CK_ALLREDUCE) {
    p.algorithm = algo;
    // the composed launch runs the twoshot all-reduce (a oneshot by
    // columns was measured slower: its N folds per column run in turn)
    if (p.algorithm == COLL_ALGO_AUTO)
      p.algorithm = path == COLL_PATH_COMPOSED ? COLL_TWOSHOT
                    : (n <= 2 || in_bytes_per_rank <= 512 * 1024) ? COLL_ONESHOT
                                                                   : COLL_TWOSHOT;
  }
  p.path = path;
  // Bounded staging (Purlin §4.1) is a mode of the composed launch: with a
  // capacity below the message, AUTO takes the composed launch and any
  // other path is refused (its kernels address the whole message).
  const bool composable = p.enc == ENC_LL128 &&
                          ((p.kind == CK_ALLREDUCE && p.algorithm == COLL_TWOSHOT) ||
                           p.kind == CK_REDUCE_SCATTER || p.kind == CK_REDUCE_SCATTER_V ||
                           p.kind == CK_ALLTOALL || p.kind == CK_ALLTOALL_V);
  const bool capped = in.staging_bytes > 0;
  if (capped && p.path == COLL_PATH_AUTO && composable) p.path = COLL_PATH_COMPOSED;
  if (p.path == COLL_PATH_AUTO) {
    if (in_bytes_per_rank <= 256 * 1024 && p.enc != ENC_LL128)
      p.path = COLL_PATH_FUSED;
    else if (p.enc == ENC_LL128 &&
             ((p.kind == CK_ALLREDUCE && p.algorithm == COLL_TWOSHOT) ||
              p.kind == CK_REDUCE_SCATTER || p.kind == CK_ALLGATHER ||
              p.kind == CK_REDUCE_SCATTER_V || p.kind == CK_ALLGATHER_V ||
              (in_bytes_per_rank >= (4u << 20) &&
               (p.kind == CK_ALLTOALL || p.kind == CK_ALLTOALL_V))))
      p.path = COLL_PATH_COMPOSED;
    else
      p.path = COLL_PATH_STREAMED;
  }

  // The composed launch: the LL128 twoshot all-reduce, reduce-scatter,
  // all-to-all and all-gather, and their V forms (stage plus one or two
  // consuming kinds of task per chunk).
  if (p.path == COLL_PATH_COMPOSED &&
      !(p.enc == ENC_LL128 &&
        ((p.kind == CK_ALLREDUCE && p.algorithm == COLL_TWOSHOT) ||
         p.kind == CK_REDUCE_SCATTER || p.kind == CK_ALLTOALL || p.kind == CK_ALLGATHER ||
         p.kind == CK_REDUCE_SCATTER_V || p.kind == CK_ALLGATHER_V ||
         p.kind == CK_ALLTOALL_V)))
    return COLL_ERR_UNSUPPORTED;

  // Rank images of region P.
  for (int r = 0; r < n; ++r) {
    std::vector<std::pair<uint64_t, uint64_t>> parts;
    if (p.kind == CK_REDUCE_SCATTER_V || p.kind == CK_ALLTOALL_V) {
      // partition k of rank r: V[k] (RS-V) or V[r][k] (A2A-V) elements,
      // packed back to back in the input
      uint64_t at = 0;
      for (int k = 0; k < n; ++k) {
        const uint64_t len = p.kind == CK_REDUCE_SCATTER_V ? V[k] : V[(size_t)r * n + k];
        parts.push_back({len, at});
        at += len;
      }
    } else if (L == COLL_SCATTERED) {
      for (int k = 0; k < n; ++k) parts.push_back({SL(k), SB(k)});
    } else {
      parts.push_back({p.in_elems[r], 0});
    }
    p.p_rank_lines = std::max<uint64_t>(p.p_rank_lines, build_image(p.enc, parts, p.pseg[r]));
  }
  const bool twoshot = p.kind == CK_ALLREDUCE && p.algorithm == COLL_TWOSHOT;
  if (twoshot) {
    for (int r = 0; r < n; ++r) {
      std::vector<std::pair<uint64_t, uint64_t>> parts{{SL(r), 0}};
      p.ag_rank_lines = std::max<uint64_t>(p.ag_rank_lines, build_image(p.enc, parts, p.agseg[r]));
    }
  }

  // CTAs per rank on the fused path: every worker CTA plus one late producer
  // per rank must be co-resident (cooperative launch).
  // By default one CTA per SM; a requested `ctas` (the option, or the policy
  // entry's launch shape) may go up to every co-resident CTA.  Always a
  // power of two per rank: the twoshot's published tiles then line up with
  // the tiles its gathers read (on GB300, 16 CTAs per rank at 8 ranks run a
  // 1 MiB twoshot in 13.5 us, 17 or 18 CTAs in 19-20 us).
  const int sms = in.sms > 0 ? in.sms : 152;
  const int cap = in.fused_capacity > 0 ? in.fused_capacity : sms;
  auto pow2_floor = [](int v) {
    v = std::max(1, v);
    while (v & (v - 1)) v &= v - 1;
    return v;
  };
  const int B_all = pow2_floor(cap / n - 1);
  int B = std::min(B_all, pow2_floor(std::min(cap, sms) / n - 1));
  if (ctas > 0) B = std::min(B_all, pow2_floor(ctas / n));

  // Tile sizes (lines, multiples of 4).
  auto fused = p.path == COLL_PATH_FUSED;
  // Streamed tiles: a 256-thread CTA moves 4 LL8 groups per thread or 4
  // LL128 rows per warp per step.
  const uint64_t max_tile = p.enc == ENC_LL128 ? 1024 : 4096;
  // Fused tiles: the smallest tile (multiple of 4 lines) that gives every
  // CTA of a rank at most one item of the phase.  When even the largest
  // tile leaves more items than CTAs, the phase takes R rounds; the tile is
  // then the smallest that fits R * B items, so every CTA gets R items of
  // about equal size (with the largest tile the last round was partial and
  // a few CTAs did twice the work of the others: an 8-rank twoshot of
  // 8 x [68 x 4096] ran at 18 us against 10 us for [64 x 4096]).
  auto pick_tile = [&](const std::vector<uint64_t>& seg_lines) -> uint64_t {
    if (in.tile_lines > 0) return round_up((uint64_t)in.tile_lines, 4);
    if (!fused) return max_tile;
    // The one-launch twoshot takes tiles of up to 16384 lines: one round of
    // larger tiles beat two balanced rounds from 128 tokens up (8 x [136 x
    // 4096]: 16.2 against 19.4 us); the oneshot keeps 4096 (larger tiles cost
    // it 5-7 % at 96-112 tokens).
    uint64_t lo = 4, hi = twoshot && p.enc != ENC_LL128 ? 16384 : max_tile;
    auto items_for = [&](uint64_t t) {
      uint64_t c = 0;
      for (uint64_t l : seg_lines) c += (l + t - 1) / t;
      return c;
    };
    const uint64_t rounds = (items_for(hi) + (uint64_t)B - 1) / (uint64_t)B;
    const uint64_t fit = std::max<uint64_t>(rounds, 1) * (uint64_t)B;
    while (lo < hi) {
      const uint64_t mid = round_up((lo + hi) / 2, 4);
      if (mid >= hi) break;
      if (items_for(mid) <= fit) hi = mid; else lo = mid + 4;
    }
    return hi;
  };
  auto seg_lines = [&](const std::vector<Seg>& segs) {
    std::vector<uint64_t> v;
    for (auto& s : segs) v.push_back(s.lines);
    return v;
  };
  // Rank images may differ (V layouts, a ragged last partition): the stage
  // tile is the largest any rank needs.
  uint64_t stile = 4;
  for (int r = 0; r < n; ++r) stile = std::max(stile, pick_tile(seg_lines(p.pseg[r])));
  const Tiler stage_tiler{stile, p.enc};
  const uint64_t epl = (uint64_t)line_elems(p.enc);

  // Stage items.
  for (int r = 0; r < n; ++r)
    for (auto& s : p.pseg[r])
      stage_tiler.over(s, [&](uint64_t t0, uint64_t nl, uint64_t ne) {
        StageItem it{};
        it.rank = (uint16_t)r;
        it.nlines = (uint32_t)nl;
        it.nelems = (uint32_t)ne;
        it.dst_line = s.line0 + t0;
        it.in_elem = s.in_elem + t0 * epl;
        p.sitems.push_back(it);
      });
  {
    int k = 0;
    for (int r = 0; r <= kMaxRanks; ++r) {
      while (k < (int)p.sitems.size() && p.sitems[k].rank < r) ++k;
      p.sbeg[r] = r <= n ? k : (int)p.sitems.size();
    }
  }

  // Consume items.
  Counters ctr;
  switch (p.kind) {
    case CK_ALLREDUCE:
      if (!twoshot) {
        // oneshot: every rank folds every partition of every rank
        const Tiler t{pick_tile(seg_lines(p.pseg[0])), p.enc};
        for (int d = 0; d < n; ++d)
          for (int k = 0; k < n; ++k) {
            const Seg& s = p.pseg[0][k];
            t.over(s, [&](uint64_t t0, uint64_t nl, uint64_t ne) {
              Item it = make_item(IK_REDUCE, d, 0, s.line0 + t0, nl, ne,
                                  SB(k) + t0 * epl);
              set_reset(it, n, ctr.get(1, s.line0 + t0));
              p.items1.push_back(it);
            });
          }
      } else {
        // twoshot phase 1: owner r folds partition r of every rank and
        // publishes it into its reduced-partition image
        const Tiler t1{pick_tile({lines_for(p.enc, M)}), p.enc};
        for (int r = 0; r < n; ++r) {
          const Seg& s = p.pseg[0][r];
          t1.over(s, [&](uint64_t t0, uint64_t nl, uint64_t ne) {
            Item it = make_item(IK_REDUCE, r, 0, s.line0 + t0, nl, ne, t0);
            it.flags |= IF_PUBLISH;
            set_reset(it, 1, 0);
            p.items1.push_back(it);
          });
        }
        // phase 2: every rank copies every owner's reduced partition
        const Tiler t2{pick_tile(std::vector<uint64_t>(n, lines_for(p.enc, M))), p.enc};
        for (int d = 0; d < n; ++d)
          for (int r = 0; r < n; ++r) {
            const Seg& s = p.agseg[r][0];
            t2.over(s, [&](uint64_t t0, uint64_t nl, uint64_t ne) {
              Item it = make_item(IK_COPY, d, r, s.line0 + t0, nl, ne,
                                  SB(r) + t0 * epl);
              set_reset(it, n, ctr.get(2, ((uint64_t)r << 40) | (s.line0 + t0)));
              p.items2.push_back(it);
            });
          }
      }
      break;
    case CK_REDUCE_SCATTER: {
      const Tiler t{pick_tile({lines_for(p.enc, M)}), p.enc};
      for (int r = 0; r < n; ++r) {
        const Seg& s = p.pseg[0][r];
        t.over(s, [&](uint64_t t0, uint64_t nl, uint64_t ne) {
          Item it = make_item(IK_REDUCE, r, 0, s.line0 + t0, nl, ne, t0 * epl);
          set_reset(it, 1, 0);
          p.items1.push_back(it);
        });
      }
      break;
    }
    case CK_ALLGATHER: {
      const Tiler t{pick_tile(std::vector<uint64_t>(n, lines_for(p.enc, M))), p.enc};
      for (int d = 0; d < n; ++d)
        for (int q = 0; q < n; ++q) {
          const Seg& s = p.pseg[q][0];
          t.over(s, [&](uint64_t t0, uint64_t nl, uint64_t ne) {
            Item it = make_item(IK_COPY, d, q, s.line0 + t0, nl, ne,
                                SB(q) + t0 * epl);
            set_reset(it, n, ctr.get(3, ((uint64_t)q << 40) | (s.line0 + t0)));
            p.items1.push_back(it);
          });
        }
      break;
    }
    case CK_ALLTOALL: {
      const Tiler t{pick_tile(std::vector<uint64_t>(n, lines_for(p.enc, M))), p.enc};
      for (int d = 0; d < n; ++d)
        for (int q = 0; q < n; ++q) {
          const Seg& s = p.pseg[q][d];
          t.over(s, [&](uint64_t t0, uint64_t nl, uint64_t ne) {
            Item it = make_item(IK_COPY, d, q, s.line0 + t0, nl, ne, (uint64_t)q * M + t0 * epl);
            set_reset(it, 1, 0);
            p.items1.push_back(it);
          });
        }
      break;
    }
    case CK_REDUCE_SCATTER_V: {
      // every rank's image has the same segments; owner r folds segment r
      std::vector<uint64_t> mine;
      for (int r = 0; r < n; ++r) mine.push_back(p.pseg[0][r].lines);
      uint64_t tile = 4;
      for (uint64_t l : mine) tile = std::max(tile, pick_tile({l}));
      const Tiler t{tile, p.enc};
      for (int r = 0; r < n; ++r) {
        const Seg& s = p.pseg[0][r];
        t.over(s, [&](uint64_t t0, uint64_t nl, uint64_t ne) {
          Item it = make_item(IK_REDUCE, r, 0, s.line0 + t0, nl, ne, t0 * epl);
          set_reset(it, 1, 0);
          p.items1.push_back(it);
        });
      }
      break;
    }
    case CK_ALLGATHER_V: {
      // every rank copies every contribution q to offset sum_{q'<q} V[q']
      std::vector<uint64_t> all;
      for (int q = 0; q < n; ++q) all.push_back(p.pseg[q][0].lines);
      const Tiler t{pick_tile(all), p.enc};
      for (int d = 0; d < n; ++d) {
        uint64_t at = 0;
        for (int q = 0; q < n; ++q) {
          const Seg& s = p.pseg[q][0];
          t.over(s, [&](uint64_t t0, uint64_t nl, uint64_t ne) {
            Item it = make_item(IK_COPY, d, q, s.line0 + t0, nl, ne, at + t0 * epl);
            set_reset(it, n, ctr.get(3, ((uint64_t)q << 40) | (s.line0 + t0)));
            p.items1.push_back(it);
          });
          at += V[q];
        }
      }
      break;
    }
    case CK_ALLTOALL_V: {
      // destination d copies segment d of every source q, in source order,
      // to offset sum_{q'<q} V[q'][d]
      uint64_t tile = 4;
      for (int d = 0; d < n; ++d) {
        std::vector<uint64_t> mine;
        for (int q = 0; q < n; ++q) mine.push_back(p.pseg[q][d].lines);
        tile = std::max(tile, pick_tile(mine));
      }
      const Tiler t{tile, p.enc};
      for (int d = 0; d < n; ++d) {
        uint64_t at = 0;
        for (int q = 0; q < n; ++q) {
          const Seg& s = p.pseg[q][d];
          t.over(s, [&](uint64_t t0, uint64_t nl, uint64_t ne) {
            Item it = make_item(IK_COPY, d, q, s.line0 + t0, nl, ne, at + t0 * epl);
            set_reset(it, 1, 0);
            p.items1.push_back(it);
          });
          at += V[(size_t)q * n + d];
        }
      }
      break;
    }
    default:
      return COLL_ERR_UNSUPPORTED;
  }
  p.ncounters = (uint32_t)ctr.keys.size();
  group_by_dst(p.items1, n, p.beg1);
  group_by_dst(p.items2, n, p.beg2);

  // Fused grid: never more CTAs per rank than the largest per-rank list.
  int most = 1;
  for (int r = 0; r < n; ++r) {
    most = std::max(most, p.sbeg[r + 1] - p.sbeg[r]);
    most = std::max(most, p.beg1[r + 1] - p.beg1[r]);
    most = std::max(most, p.beg2[r + 1] - p.beg2[r]);
  }
  p.ctas_per_rank = std::max(1, std::min(B, most));
  const int consume_cap = in.ctas > 0 ? in.ctas : sms * 8;
  p.consume_grid = std::max(1, std::min<int>(consume_cap, (int)std::max(p.items1.size(), p.items2.size())));

  // Workspace layout.
  uint64_t off = sizeof(WsHeader);
  off = round_up(off, 256);
  p.off_sitems = off;
  off = round_up(off + p.sitems.size() * sizeof(StageItem), 256);
  p.off_items1 = off;
  off = round_up(off + p.items1.size() * sizeof(Item), 256);
  p.off_items2 = off;
  off = round_up(off + p.items2.size() * sizeof(Item), 256);
  p.off_counters = off;
  off = round_up(off + (uint64_t)std::max<uint32_t>(p.ncounters, 1) * 4, 256);
  if (p.path == COLL_PATH_COMPOSED) {
    uint64_t most = 0;
    for (int r = 0; r < n; ++r)
      for (const Seg& sg : p.pseg[r]) most = std::max<uint64_t>(most, sg.lines);
    p.composed_max_chunks = std::max<uint64_t>(1, (most + kComposedMinChunk - 1) / kComposedMinChunk);
    p.off_cflags = off;
    off += p.composed_max_chunks * ((uint64_t)n * 16 + 8);
    if (p.kind == CK_ALLTOALL || p.kind == CK_ALLTOALL_V) {
      // source q's partition d goes to destination d after the partitions
      // d of sources 0 .. q-1
      p.exch.assign((size_t)n * n, ExchPiece{});
      for (int d = 0; d < n; ++d) {
        uint64_t at = 0;
        for (int q = 0; q < n; ++q) {
          const Seg& sg = p.pseg[q][d];
          p.exch[(size_t)q * n + d] = ExchPiece{sg.line0, sg.elems, sg.in_elem, at};
          at += sg.elems;
        }
      }
      off = round_up(off, 256);
      p.off_exch = off;
      off += p.exch.size() * sizeof(ExchPiece);
    }
  }
  off = round_up(off, 4096);
  const uint64_t lb = (uint64_t)line_bytes(p.enc);
  if (capped && in.staging_bytes < p.p_rank_lines * lb) {
    // cycling needs the composed launch of a collective whose chunk slots
    // hold all N partitions of a chunk (not the all-gather's one segment)
    if (p.path != COLL_PATH_COMPOSED || !composable) return COLL_ERR_UNSUPPORTED;
    // chunk slots of N partitions x chunk lines; at least two slots of the
    // smallest chunk
    p.ring_lines = in.staging_bytes / lb / ((uint64_t)n * kComposedMinChunk) *
                   ((uint64_t)n * kComposedMinChunk);
    if (p.ring_lines < 2ull * n * kComposedMinChunk) return COLL_ERR_INVALID;
    p.p_rank_lines = p.ring_lines;
    if (p.ag_rank_lines > 0) p.ag_rank_lines = std::min(p.ag_rank_lines, p.ring_lines / n);
  }
  p.P.rank_bytes = round_up(p.p_rank_lines * lb, 4096);
  p.P.slot_bytes = p.P.rank_bytes * (uint64_t)n;
  p.P.slot_mask = (uint64_t)p.slots - 1;
  p.P.base = off;
  off += (uint64_t)p.slots * p.P.slot_bytes;
  p.AG.rank_bytes = round_up(p.ag_rank_lines * lb, 4096);
  p.AG.slot_bytes = p.AG.rank_bytes * (uint64_t)n;
  p.AG.slot_mask = (uint64_t)p.slots - 1;
  p.AG.base = off;
  off += (uint64_t)p.slots * p.AG.slot_bytes;
  p.ws_bytes = off;
  // Dependent launches overlap each kernel's launch with the tail of the one
  // before it.  8 ranks, warm, per op: one launch 3.94 -> 3.59 us at 8 KiB,
  // 10.78 -> 10.43 us at 512 KiB, but 12.88 -> 13.75 us at 1 MiB; stream-
  // ordered oneshot 5.37 -> 4.54 us at 8 KiB, 11.94 -> 11.31 us at 128 KiB,
  // but 16.94 -> 18.54 us at 512 KiB and 75.8 -> 81.6 us for the twoshot at
  // 4 MiB.  So: one-launch runs up to 512 KiB per rank (input or output),
  // stream-ordered ones up to 128 KiB.  The composed launch by columns: up
  // to 512 KiB too (8 ranks, all-reduce, 16 KiB / 128 KiB / 512 KiB: 7.35
  // -> 6.80, 7.89 -> 7.25, 8.00 -> 7.43 us), not at 1 MiB (9.74 -> 11.51).
  uint64_t largest = 0;
  for (int r = 0; r < n; ++r)
    largest = std::max(largest, std::max(p.in_elems[r], p.out_elems[r]));
  const uint64_t bytes = largest * 2;
  p.dependent_launch =
      ((p.path == COLL_PATH_FUSED || p.path == COLL_PATH_COMPOSED) && bytes <= 512 * 1024) ||
      (p.path == COLL_PATH_STREAMED && bytes <= 128 * 1024);
  return COLL_OK;
}

}  // namespace coll
