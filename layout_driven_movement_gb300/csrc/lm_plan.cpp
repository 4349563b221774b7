// Lowering of a src/dst layout pair into a copy plan.
//
// 1. Both layouts are split over the same logical domain into joint modes
//    (extent, src stride, dst stride): the common refinement of their leaf
//    lists.  The copy out[dst(i)] = in[src(i)] is a set of (src, dst) offset
//    pairs, so the order of the joint modes is free; modes that continue one
//    another on both sides are merged ("coalescing").
// 2. The destination must be one-to-one (two logical indices writing one
//    slot would leave the result undefined).
// 3. A mode with unit stride on both sides is the common contiguous run --
//    the common vector of the inverse layouts ("CUTE布局代数" §2.3); when it
//    spans 16 bytes the VEC kernel moves 16-byte vectors directly.
// 4. Otherwise, when the source has a unit-stride mode and the destination
//    has one, the STAGED kernel copies tiles: loads run along the source's
//    contiguous modes, stores along the destination's, and the tile passes
//    through shared memory laid out with an XOR swizzle chosen here by
//    simulating the bank conflicts of both phases ("CUTLASS Layout可视化" §5.2
//    and §4.3: spread one warp's accesses over the 32 banks; the
//    PitchLinearStripminedThreadMap article §4.1: 128-byte lines).
// 5. Everything else runs GENERIC: one element per thread.

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <numeric>
#include <sstream>

#include "lm_internal.h"

namespace lm {

bool refine(const std::vector<Leaf>& a, const std::vector<Leaf>& b,
            std::vector<JMode>& out);  // lm_layout.cpp

namespace {

constexpr int64_t kSmall = 4096;            // elements: GENERIC below this
constexpr int64_t kMaxPiece = int64_t(1) << 31;
constexpr int kThreads = 256;               // STAGED block size

int ilog2(int64_t v) {
  int l = 0;
  while ((int64_t(1) << l) < v) ++l;
  return l;
}

Swz to_bytes(const Swz& z, int eb) {
  if (!z.on()) return Swz{};
  return Swz{z.b, z.m + ilog2(eb), z.s};
}

int64_t prod_e(const std::vector<JMode>& ms) {
  int64_t p = 1;
  for (const JMode& m : ms) p = mul_chk(p, m.e);
  return p;
}

std::vector<JMode> coalesce_joint(std::vector<JMode> ms) {
  ms.erase(std::remove_if(ms.begin(), ms.end(),
                          [](const JMode& m) { return m.e == 1; }),
           ms.end());
  bool merged = true;
  while (merged) {
    merged = false;
    for (size_t i = 0; i < ms.size() && !merged; ++i)
      for (size_t j = 0; j < ms.size() && !merged; ++j) {
        if (i == j) continue;
        if (ms[j].s == ms[i].e * ms[i].s && ms[j].d == ms[i].e * ms[i].d) {
          ms[i].e = mul_chk(ms[i].e, ms[j].e);
          ms.erase(ms.begin() + long(j));
          merged = true;
        }
      }
  }
  return ms;
}

// ---------------------------------------------------------------------------
// GENERIC
// ---------------------------------------------------------------------------

void fill_side(const std::vector<Leaf>& ls, int eb, uint32_t* ext,
               FastDiv* div, int64_t* str, int64_t* ext64, int32_t& n) {
  std::vector<Leaf> c;
  for (const Leaf& l : ls)
    if (l.e != 1) c.push_back(l);
  if (c.size() > size_t(kMaxLeaves)) fail(LM_E_NOT_REPRESENTABLE);
  n = int32_t(c.size());
  for (size_t k = 0; k < c.size(); ++k) {
    ext64[k] = c[k].e;
    ext[k] = c[k].e < (int64_t(1) << 31) ? uint32_t(c[k].e) : 0u;
    div[k] = make_fastdiv(ext[k] ? ext[k] : 1u);
    str[k] = mul_chk(c[k].d, eb);
  }
}

GenericArgs make_generic(const std::vector<Leaf>& sl,
                         const std::vector<Leaf>& dl, int64_t n,
                         int64_t s_base, int64_t d_base, const Swz& ss,
                         const Swz& ds, int eb) {
  GenericArgs g;
  g.n = uint64_t(n);
  g.eb = eb;
  g.wide = n >= (int64_t(1) << 31) ? 1 : 0;
  fill_side(sl, eb, g.s_ext, g.s_div, g.s_str, g.s_ext64, g.ns);
  fill_side(dl, eb, g.d_ext, g.d_div, g.d_str, g.d_ext64, g.nd);
  for (int k = 0; k < g.ns; ++k)
    if (!g.s_ext[k]) g.wide = 1;
  for (int k = 0; k < g.nd; ++k)
    if (!g.d_ext[k]) g.wide = 1;
  g.s_base = mul_chk(s_base, eb);
  g.d_base = mul_chk(d_base, eb);
  g.s_swz = to_bytes(ss, eb);
  g.d_swz = to_bytes(ds, eb);
  return g;
}

int env_int(const char* name, int dflt);

// Tiled form of a copy without a common refinement (GTileArgs), when one
// side's first leaf has unit stride and at least kGtU coordinates and the
// other side's unit-stride leaf, of at least kGtU coordinates, sits behind
// leaves spanning at least kGtU indices.  LM_GTILE=0 keeps one element per
// thread.
bool plan_gtile(const std::vector<Leaf>& sl, const std::vector<Leaf>& dl,
                int64_t n, const Swz& ss, const Swz& ds, int eb,
                GTileArgs& g) {
  static const bool on = env_int("LM_GTILE", 1) != 0;
  if (!on || n < 1 || n >= (int64_t(1) << 32)) return false;
  auto unit_leaf = [](const std::vector<Leaf>& L) {
    for (size_t k = 0; k < L.size(); ++k)
      if (L[k].d == 1) return int(k);
    return -1;
  };
  const int ks = unit_leaf(sl), kd = unit_leaf(dl);
  bool outer_src;
  if (kd == 0 && ks > 0)
    outer_src = true;
  else if (ks == 0 && kd > 0)
    outer_src = false;
  else
    return false;
  const std::vector<Leaf>& outer = outer_src ? sl : dl;
  const std::vector<Leaf>& inner = outer_src ? dl : sl;
  const int k = outer_src ? ks : kd;
  int64_t W = 1;
  for (int j = 0; j < k; ++j) W *= outer[size_t(j)].e;
  if (W < kGtU || inner[0].e < kGtU || outer[size_t(k)].e < kGtU) return false;
  if (k > kGtLeaves || int(outer.size()) - k > kGtLeaves ||
      int(inner.size()) > kGtLeaves)
    return false;
  g = GTileArgs{};
  g.n = uint64_t(n);
  g.W = uint32_t(W);
  g.nv = uint32_t(n / W);
  // tiles of 64 along u when u runs that far (LM_GTILE_U=32 keeps 32)
  static const int tu_env = env_int("LM_GTILE_U", 64);
  g.tile_u = tu_env == 32 || W < 64 ? 32u : 64u;
  g.n_ut = uint32_t((W + g.tile_u - 1) / g.tile_u);
  g.n_vt = uint32_t((int64_t(g.nv) + kGtV - 1) / kGtV);
  g.ut_div = make_fastdiv(g.n_ut);
  g.outer_src = outer_src ? 1 : 0;
  for (int j = 0; j < int(outer.size()); ++j) {
    const Leaf& l = outer[size_t(j)];
    if (j < k) {
      g.lo_ext[g.n_lo] = uint32_t(l.e);
      g.lo_div[g.n_lo] = make_fastdiv(uint32_t(l.e));
      g.lo_str[g.n_lo++] = mul_chk(l.d, eb);
    } else {
      g.hi_ext[g.n_hi] = uint32_t(l.e);
      g.hi_div[g.n_hi] = make_fastdiv(uint32_t(l.e));
      g.hi_str[g.n_hi++] = mul_chk(l.d, eb);
    }
  }
  for (const Leaf& l : inner) {
    g.in_ext[g.n_in] = uint32_t(l.e);
    g.in_div[g.n_in] = make_fastdiv(uint32_t(l.e));
    g.in_str[g.n_in++] = mul_chk(l.d, eb);
  }
  // the steps as digits (colex)
  auto digits = [](int64_t x, const uint32_t* ext, int n, uint32_t* out) {
    for (int j = 0; j < n; ++j) {
      out[j] = uint32_t(x % ext[j]);
      x /= ext[j];
    }
  };
  // a step's offset change without carries, and each leaf's carry change
  auto dstep = [](const uint32_t* d, const int64_t* str, int n) {
    int64_t r = 0;
    for (int j = 0; j < n; ++j) r = add_chk(r, mul_chk(int64_t(d[j]), str[j]));
    return r;
  };
  auto cadj = [](const uint32_t* ext, const int64_t* str, int n,
                 int64_t* out) {
    for (int j = 0; j < kMaxLeaves; ++j)
      out[j] = j + 1 < n ? add_chk(str[j + 1], -mul_chk(int64_t(ext[j]),
                                                        str[j]))
                         : 0;
  };
  cadj(g.lo_ext, g.lo_str, g.n_lo, g.lo_cadj);
  cadj(g.in_ext, g.in_str, g.n_in, g.in_cadj);
  // lanes over v: 256 / kGtV rows of u per pass; lanes over u:
  // 256 / tile_u columns of v per pass
  digits(256 / kGtV, g.lo_ext, g.n_lo, g.lo_step);
  digits(int64_t(256 / g.tile_u) * W, g.in_ext, g.n_in, g.in_step);
  g.lo_dstep = dstep(g.lo_step, g.lo_str, g.n_lo);
  g.in_dstep = dstep(g.in_step, g.in_str, g.n_in);
  // tensor-map loads (LM_GTILE_TMA=0 keeps cp.async): the source outer, a
  // plain matrix (one leaf on each side of its unit-stride leaf), rows
  // 16-byte aligned, 2- to 8-byte elements, no source swizzle, 64-row tiles
  static const bool tma_on = env_int("LM_GTILE_TMA", 1) != 0;
  if (tma_on && outer_src && !ss.on() && g.n_lo == 1 && g.n_hi == 1 &&
      g.tile_u == 64 && (eb == 2 || eb == 4 || eb == 8) &&
      g.lo_str[0] % 16 == 0 && g.lo_str[0] > 0 &&
      g.lo_str[0] < (int64_t(1) << 40) && g.n_in <= 2 && g.nv >= 64 &&
      W >= 64) {
    const uint32_t vpc = uint32_t(16 / eb);       // v per 16-byte chunk
    const uint32_t cp = 256u / g.tile_u;          // chunks a pass spans
    g.tma = 1;
    g.t_vpr = uint32_t(128 / eb);
    g.t_regions = uint32_t(kGtV) / g.t_vpr;
    g.t_ustride = g.lo_str[0];
    digits(W, g.in_ext, g.n_in, g.in_step1);
    digits(int64_t(cp * vpc - vpc + 1) * W, g.in_ext, g.n_in, g.in_jump);
    g.in_dstep1 = dstep(g.in_step1, g.in_str, g.n_in);
    g.in_djump = dstep(g.in_jump, g.in_str, g.n_in);
  }
  // 32-bit offsets when every offset of both sides, swizzled or not, stays
  // below 2^31 bytes
  auto reach = [&](const std::vector<Leaf>& L, const Swz& z) {
    int64_t r = 0;
    for (const Leaf& l : L) r = add_chk(r, mul_chk(l.e - 1, l.d));
    r = mul_chk(add_chk(r, 1), eb);
    if (z.on()) r = add_chk(r, int64_t(eb) << (z.b + z.m + z.s));
    return r;
  };
  // ... and so does every step's offset change (32-bit arithmetic)
  auto small = [](int64_t x) {
    return x > -(int64_t(1) << 31) && x < (int64_t(1) << 31);
  };
  bool steps32 = small(g.lo_dstep) && small(g.in_dstep) &&
                 small(g.in_dstep1) && small(g.in_djump);
  for (int j = 0; j < kMaxLeaves; ++j)
    steps32 = steps32 && small(g.lo_cadj[j]) && small(g.in_cadj[j]);
  g.narrow = reach(sl, ss) < (int64_t(1) << 31) &&
                     reach(dl, ds) < (int64_t(1) << 31) && steps32
                 ? 1
                 : 0;
  g.s_swz = to_bytes(ss, eb);
  g.d_swz = to_bytes(ds, eb);
  return true;
}

GenericArgs generic_for_modes(const std::vector<JMode>& ms, int64_t s_base,
                              int64_t d_base, const lm_plan& P) {
  std::vector<Leaf> sl, dl;
  for (const JMode& m : ms) {
    sl.push_back({m.e, m.s});
    dl.push_back({m.e, m.d});
  }
  return make_generic(sl, dl, prod_e(ms), s_base, d_base, P.s_swz, P.d_swz,
                      P.eb);
}

// ---------------------------------------------------------------------------
// STAGED: tile choice, chains, smem layout search
// ---------------------------------------------------------------------------

struct TileMode {
  int mode;     // index into the piece's joint modes
  int64_t T;    // tile extent along it (divides the mode's extent)
};

// LM_TRANSPOSE=0 plans 2-D transposes with the per-element gather store
// instead of register micro-tiles (for comparing the two).
bool transpose_disabled() {
  static bool v = [] {
    const char* e = std::getenv("LM_TRANSPOSE");
    return e && e[0] == '0';
  }();
  return v;
}

int env_int(const char* name, int dflt) {
  const char* e = std::getenv(name);
  return e ? std::atoi(e) : dflt;
}
// cp.async pipeline depth of STAGED kernels (LM_STAGES, 2 or 3)
int staged_stages() {
  static int v = env_int("LM_STAGES", 2) == 3 ? 3 : 2;
  return v;
}
// 16-byte vectors per thread per tile of the tiled VEC kernel
// (LM_VEC_UNROLL, 4 or 8)
int vec_unroll() {
  static int v = env_int("LM_VEC_UNROLL", 4) == 8 ? 8 : 4;
  return v;
}

// Bulk-copy (TMA) loads for STAGED tiles (LM_BULK=0 turns them off) and
// their pipeline depth (LM_BULK_STAGES, 2..4).
bool bulk_enabled() {
  static bool v = env_int("LM_BULK", 1) != 0;
  return v;
}
int bulk_stages() {
  static int v = std::clamp(env_int("LM_BULK_STAGES", 2), 2, 4);
  return v;
}
// Tensor-map (TMA) tile loads for STAGED transposes (LM_TMA=1 turns them
// on) and their pipeline depth (LM_TMA_STAGES, 2..4).  Off by default:
// measured on GB300, one dense box per tile (64 rows of 256 bytes) took
// 29.3 us for the 4096x4096 fp32 transpose and 41.6 us for NHWC->NCHW
// against 23.2 and 33.4 us for the per-thread cp.async loads, whatever the
// depth, tiles per block or micro-tile order (ncu: the L1 pipeline 78%
// busy with scattered stores or conflicting shared reads); with 128-byte
// swizzled boxes and warp-block micro-tiles the fp32 transpose took 25.2 us.
bool tma_enabled() {
  static bool v = env_int("LM_TMA", 0) != 0;
  return v;
}
int tma_stages() {
  static int v = std::clamp(env_int("LM_TMA_STAGES", 3), 2, 4);
  return v;
}
// Bulk copies pay off for long rows: the bf16/fp32 transposes' 128-256 byte
// rows ran faster with per-thread cp.async (measured on GB300), the 9 KiB
// segments of the padded TV gather faster with one bulk copy.
constexpr int64_t kBulkMinSegment = 1024;

// Largest byte offset + 1 the loads of any tile reach from the buffer start.
int64_t src_reach(const StagedArgs& A) {
  int64_t r = add_chk(A.s_base, int64_t(A.seg_bytes));
  for (int k = 0; k < A.ng; ++k)
    r = add_chk(r, mul_chk(int64_t(A.g_ext[k]) - 1, A.g_s[k]));
  for (int k = 0; k < A.nso; ++k)
    r = add_chk(r, mul_chk(int64_t(A.so_ext[k]) - 1, A.so_s[k]));
  return r;
}

// Order of the tile grid (and of the VEC modes): by destination stride
// (LM_GRID_ORDER=d, default) or by source stride (LM_GRID_ORDER=s).
bool order_by_src() {
  static bool v = [] {
    const char* e = std::getenv("LM_GRID_ORDER");
    return e && e[0] == 's';
  }();
  return v;
}
bool mode_before(const JMode& x, const JMode& y) {
  return order_by_src() ? (x.s < y.s || (x.s == y.s && x.d < y.d))
                        : (x.d < y.d || (x.d == y.d && x.s < y.s));
}
// Bytes of one shared-memory row (along the source-fast mode) of a
// transpose tile (LM_XPOSE_ROW_BYTES, default 256).
int64_t xpose_row_bytes() {
  static int64_t v = std::clamp(env_int("LM_XPOSE_ROW_BYTES", 256), 64, 4096);
  return v;
}

int64_t tile_bytes_target() {
  static int64_t v = [] {
    const char* e = std::getenv("LM_TILE_BYTES");
    int64_t t = e ? std::atoll(e) : 16384;
    return std::clamp<int64_t>(t, 1024, 24576);
  }();
  return v;
}

// Largest divisor of e that is <= want and a multiple of `mult`, or 0.
int64_t divisor_at_most(int64_t e, int64_t want, int64_t mult) {
  want = std::min(want, e);
  for (int64_t t = want; t >= 1; --t)
    if (e % t == 0 && t % mult == 0) return t;
  return 0;
}

// Wavefronts of one warp-wide shared-memory instruction: per phase (lanes
// whose requests share one 128-byte pass), the largest number of distinct
// 4-byte words any of the 32 banks must deliver.
int64_t wavefronts(const int64_t* addr, const bool* valid, int lanes,
                   int bytes) {
  const int per_phase = bytes <= 4 ? 32 : 128 / bytes;
  const int words = bytes <= 4 ? 1 : bytes / 4;
  int64_t total = 0;
  for (int p0 = 0; p0 < lanes; p0 += per_phase) {
    int64_t seen[32][32];
    int cnt[32] = {0};
    int worst = 0;
    bool any = false;
    for (int l = p0; l < std::min(lanes, p0 + per_phase); ++l) {
      if (!valid[l]) continue;
      any = true;
      for (int w = 0; w < words; ++w) {
        const int64_t word = (addr[l] >> 2) + w;
        const int bank = int(word & 31);
        bool dup = false;
        for (int q = 0; q < cnt[bank]; ++q)
          if (seen[bank][q] == word) dup = true;
        if (!dup && cnt[bank] < 32) seen[bank][cnt[bank]++] = word;
        worst = std::max(worst, cnt[bank]);
      }
    }
    if (any) total += std::max(worst, 1);
  }
  return total;
}


// The shared-memory image of a tile: n_seg segments of seg_bytes, placed at a
// pitch of seg_bytes + pad, then XOR-swizzled in 16-byte units.  Loads write
// 16-byte chunks; the store side reads `per` accesses of `width` bytes for
// each of n_reads slots.  Chooses the pad and swizzle with the fewest
// simulated wavefronts over every warp of one tile.
struct SmemLayout {
  int64_t pad = 0;
  Swz z;
  int64_t bytes = 0, cost = -1, ideal = 0;
  int64_t read_cost = 0, read_ideal = 0;  // the store side's reads alone
};

// LM_SMEM_SEARCH=0 keeps the plain image (no pad, no swizzle): a tuning and
// validation knob that shows the conflicts the search removes.
bool smem_search_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("LM_SMEM_SEARCH");
    return !(v && v[0] == '0');
  }();
  return on;
}

template <class ReadAddr>
SmemLayout search_smem(int threads, int64_t n_seg, int64_t seg_bytes,
                       int64_t n_reads, int per, int width,
                       const ReadAddr& read_addr, bool allow_swizzle = true,
                       bool allow_pad = true) {
  SmemLayout best;
  const int64_t cps = seg_bytes / 16;
  const int64_t n_l = n_seg * cps;
  const int64_t lpt = (n_l + threads - 1) / threads;
  const int64_t spt = (n_reads + threads - 1) / threads;
  const bool search = smem_search_enabled();
  const std::vector<int64_t> pads =
      n_seg > 1 && search && allow_pad
          ? std::vector<int64_t>{0, 16, 32, 48, 64, 80, 96, 112}
          : std::vector<int64_t>{0};
  std::vector<Swz> zs{Swz{}};
  if (allow_swizzle && search)
    for (int bb = 1; bb <= 3; ++bb)
      for (int ss = bb; ss <= 10; ++ss) zs.push_back(Swz{bb, 4, ss});
  std::vector<int64_t> addr(32);
  bool valid[32];
  for (int64_t pad : pads) {
    const int64_t pitch = seg_bytes + pad;
    const int64_t lin_max = (n_seg - 1) * pitch + seg_bytes;
    for (const Swz& z : zs) {
      const int64_t blk = int64_t(16) << z.b;
      const int64_t bytes = ((lin_max + blk - 1) / blk) * blk;
      if (bytes > 24576) continue;
      int64_t cost = 0, id = 0, rcost = 0, rid = 0;
      for (int w = 0; w < threads / 32; ++w) {
        for (int64_t k = 0; k < lpt; ++k) {
          int cnt = 0;
          for (int l = 0; l < 32; ++l) {
            const int64_t j = 32 * w + l + k * threads;
            valid[l] = j < n_l;
            cnt += valid[l];
            addr[size_t(l)] =
                valid[l] ? z.apply((j / cps) * pitch + (j % cps) * 16) : 0;
          }
          cost += wavefronts(addr.data(), valid, 32, 16);
          id += (cnt * 16 + 127) / 128;
        }
        for (int64_t k = 0; k < spt; ++k)
          for (int e = 0; e < per; ++e) {
            int cnt = 0;
            for (int l = 0; l < 32; ++l) {
              const int64_t j = 32 * w + l + k * threads;
              valid[l] = j < n_reads;
              cnt += valid[l];
              addr[size_t(l)] = valid[l] ? z.apply(read_addr(j, e, pitch)) : 0;
            }
            rcost += wavefronts(addr.data(), valid, 32, width);
            rid += cnt ? (cnt * width + 127) / 128 : 0;
          }
      }
      cost += rcost;
      id += rid;
      if (best.cost < 0 || cost < best.cost ||
          (cost == best.cost && bytes < best.bytes)) {
        best.pad = pad;
        best.z = z;
        best.cost = cost;
        best.bytes = bytes;
        best.ideal = id;
        best.read_cost = rcost;
        best.read_ideal = rid;
      }
    }
  }
  return best;
}

}  // namespace

int64_t warp_wavefronts(const int64_t* addr, const bool* valid, int bytes) {
  return wavefronts(addr, valid, 32, bytes);
}

// A common refinement of the two sides' leaves, trying each side's leaves
// as given and coalesced: coalescing keeps a side's offset function (it
// only merges leaves that continue each other), but removes boundaries the
// other side does not share -- (6000,7000):(7000,1) against
// (7000,6000):(1,7000) refines only once the second side is seen as the
// single run 42000000:1.
bool refine_sides(const std::vector<Leaf>& s, const std::vector<Leaf>& d,
                  std::vector<JMode>& out) {
  if (refine(s, d, out)) return true;
  const std::vector<Leaf> cs = coalesce_leaves(s), cd = coalesce_leaves(d);
  return refine(cs, d, out) || refine(s, cd, out) || refine(cs, cd, out);
}

bool joint_modes(const lm_layout& src, const lm_layout& dst,
                 std::vector<JMode>& out) {
  out.clear();
  if (!refine_sides(src.leaves, dst.leaves, out)) return false;
  out = coalesce_joint(out);
  return true;
}

namespace {

struct StagedChoice {
  bool ok = false;
  int split_mode = -1;     // > = 0: split the box along this mode at split_at
  int64_t split_at = 0;
};

}  // namespace

// Grid over tiles (colex, fastest first) and the piece's global placement.
static void fill_grid(StagedArgs& A, const std::vector<JMode>& grid,
                      int64_t s_base, int64_t d_base, int eb, const Swz& ssb,
                      const Swz& dsb) {
  A.n_tiles = uint32_t(prod_e(grid));
  A.ng = int32_t(grid.size());
  uint32_t pre = 1;
  for (size_t k = 0; k < grid.size(); ++k) {
    A.g_ext[k] = uint32_t(grid[k].e);
    A.g_pre[k] = make_fastdiv(pre);
    A.g_div[k] = make_fastdiv(uint32_t(grid[k].e));
    A.g_s[k] = mul_chk(grid[k].s, eb);
    A.g_d[k] = mul_chk(grid[k].d, eb);
    pre *= uint32_t(grid[k].e);
  }
  A.s_base = mul_chk(s_base, eb);
  A.d_base = mul_chk(d_base, eb);
  A.s_swz = ssb;
  A.d_swz = dsb;
}

// Bytes per tile for a box of `total_bytes`: 16 KiB, smaller for small boxes
// so that there are at least ~8 tiles per SM (152 SMs) to balance.
static int64_t tile_target(int64_t total_bytes) {
  int64_t t = 16384;
  while (t > 2048 && total_bytes / t < 152 * 8) t /= 2;
  return t;
}

static int64_t load_reach(const StagedArgs& A, int64_t seg_bytes) {
  int64_t r = seg_bytes;
  for (int k = 0; k < A.nso; ++k)
    r = add_chk(r, mul_chk(int64_t(A.so_ext[k]) - 1, A.so_s[k]));
  return r;
}

// STAGED with the transpose store.  The tile is T_a x T_b over the src-fast
// mode a (unit source stride) and the dst-fast mode b (unit destination
// stride); the shared-memory image holds one row of T_a elements per b.
// Micro-tiles are R rows by one 16-byte chunk: R = V when b's runs hold
// whole 16-byte vectors, or R = extent(b) < V when b is short and a
// continues its destination run (an interleave).
// LM_ZIP=0 keeps short interleaves on the shared-memory transpose.
static bool zip_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("LM_ZIP");
    return !(v && v[0] == '0');
  }();
  return on;
}

// The in-register interleave: the destination-fast mode b is short (R
// coordinates, destination stride 1) and the source-fast mode a continues
// it in the destination (stride R).  Vector j of a names R source vectors
// (b's rows) and R consecutive destination vectors; no shared memory.
static bool plan_zip(const std::vector<JMode>& ms, int a, int b, int64_t R,
                     int64_t s_base, int64_t d_base, const lm_plan& P,
                     Piece& pc) {
  const int64_t eb = P.eb, V = 16 / eb;
  const JMode ma = ms[size_t(a)], mb = ms[size_t(b)];
  auto al = [](int64_t bytes) { return bytes % 16 == 0; };
  if (ma.e % V || ma.d != R || mb.d != 1 || mb.e != R) return false;
  if (!al(s_base * eb) || !al(d_base * eb) || !al(mb.s * eb)) return false;
  std::vector<JMode> rest;
  for (int k = 0; k < int(ms.size()); ++k) {
    if (k == a || k == b) continue;
    if (!al(ms[size_t(k)].s * eb) || !al(ms[size_t(k)].d * eb)) return false;
    rest.push_back(ms[size_t(k)]);
  }
  if (rest.size() + 1 > size_t(kMaxModes)) return false;
  std::sort(rest.begin(), rest.end(), mode_before);
  const int64_t nvec = prod_e(ms) / (V * R);
  if (nvec >= (int64_t(1) << 32)) return false;
  VecArgs& A = pc.vec;
  A = VecArgs{};
  A.n_vec = uint32_t(nvec);
  A.nm = int32_t(rest.size() + 1);
  A.ext[0] = uint32_t(ma.e / V);
  A.div[0] = make_fastdiv(A.ext[0]);
  A.s[0] = 16;
  A.d[0] = 16 * R;
  for (size_t k = 0; k < rest.size(); ++k) {
    A.ext[k + 1] = uint32_t(rest[k].e);
    A.div[k + 1] = make_fastdiv(A.ext[k + 1]);
    A.s[k + 1] = mul_chk(rest[k].s, eb);
    A.d[k + 1] = mul_chk(rest[k].d, eb);
  }
  A.s_base = mul_chk(s_base, eb);
  A.d_base = mul_chk(d_base, eb);
  A.zip_rows = int32_t(R);
  A.zip_s_row = mul_chk(mb.s, eb);
  pc.vec_bytes = 16;
  pc.path = PATH_ZIP;
  pc.xr = int(R);
  return true;
}

static StagedChoice plan_transpose(const std::vector<JMode>& ms,
                                   int64_t s_base, int64_t d_base,
                                   const lm_plan& P, Piece& pc) {
  StagedChoice ch;
  const int eb = P.eb;
  if (eb > 8) return ch;
  const int64_t V = 16 / eb;
  const int n = int(ms.size());
  int a = -1, b = -1;
  for (int k = 0; k < n; ++k) {
    if (ms[size_t(k)].s == 1 && a < 0) a = k;
    if (ms[size_t(k)].d == 1 && b < 0) b = k;
  }
  if (a < 0 || b < 0 || a == b) return ch;
  const Swz ssb = to_bytes(P.s_swz, eb), dsb = to_bytes(P.d_swz, eb);
  if ((ssb.on() && ssb.m < 4) || (dsb.on() && dsb.m < 4)) return ch;
  const JMode ma = ms[size_t(a)], mb = ms[size_t(b)];
  int64_t R;
  if (mb.e >= V) {
    R = V;
  } else if (V % mb.e == 0 && ma.d == mb.e) {
    R = mb.e;
  } else {
    return ch;
  }
  // ragged extents: split off the tail that is not a whole chunk/vector
  if (ma.e % V) {
    if (ma.e >= 2 * V) {
      ch.split_mode = a;
      ch.split_at = ma.e - ma.e % V;
    }
    return ch;
  }
  if (R == V && mb.e % V) {
    if (mb.e >= 2 * V) {
      ch.split_mode = b;
      ch.split_at = mb.e - mb.e % V;
    }
    return ch;
  }
  if (R < V && zip_enabled() && !ssb.on() && !dsb.on() &&
      plan_zip(ms, a, b, R, s_base, d_base, P, pc)) {
    ch.ok = true;
    return ch;
  }
  const int64_t target = tile_target(mul_chk(prod_e(ms), eb)) / eb;
  int64_t Ta, Tb;
  if (R == V) {
    Ta = divisor_at_most(ma.e, std::max<int64_t>(V, xpose_row_bytes() / eb), V);
    if (!Ta) return ch;
    const int64_t want_b = std::max<int64_t>(V, target / Ta);
    Tb = divisor_at_most(mb.e, want_b, V);
    if (Tb * 2 <= want_b && mb.e > want_b) {
      int64_t w = V;
      while (w * 2 <= want_b) w *= 2;
      if (mb.e % w) {
        ch.split_mode = b;
        ch.split_at = mb.e - mb.e % w;
        return ch;
      }
      Tb = w;
    }
  } else {
    Tb = mb.e;
    const int64_t want_a = std::max<int64_t>(V, target / Tb);
    Ta = divisor_at_most(ma.e, want_a, V);
    if (Ta * 2 <= want_a && ma.e > want_a) {
      int64_t w = V;
      while (w * 2 <= want_a) w *= 2;
      if (ma.e % w) {
        ch.split_mode = a;
        ch.split_at = ma.e - ma.e % w;
        return ch;
      }
      Ta = w;
    }
  }
  const int64_t n_bc = Tb / R, n_ac = Ta / V;
  const int64_t n_micro = n_bc * n_ac;
  const int64_t seg_bytes = Ta * eb;
  const int64_t cps = seg_bytes / 16;
  // one micro-tile per thread where possible; enough threads for the loads
  // (these limits match XposeStore: micro-tiles and load chunks per thread)
  const int64_t max_m = R >= 8 ? 1 : 2, max_l = R >= 8 ? 8 : 4;
  auto r32 = [](int64_t v) { return ((v + 31) / 32) * 32; };
  const int64_t threads = std::clamp<int64_t>(
      std::max(r32(std::min<int64_t>(n_micro, 256)),
               r32((Tb * cps + max_l - 1) / max_l)),
      32, 256);
  if (n_micro > max_m * threads || Tb * cps > threads * max_l) return ch;

  // alignment of every 16-byte access
  auto al = [&](int64_t elems) { return (elems * eb) % 16 == 0; };
  if (!al(s_base) || !al(d_base) || !al(mb.s)) return ch;
  if (R == V && !al(ma.d)) return ch;
  // the tensor dimension of each joint mode for tensor-map loads: a, b,
  // then the rest in order
  std::vector<int> tdim(size_t(n), 0);
  {
    int next = 2;
    for (int k = 0; k < n; ++k)
      tdim[size_t(k)] = k == a ? 0 : (k == b ? 1 : next++);
  }
  struct GridMode {
    JMode m;
    int tdim;
    int64_t tstep;
  };
  std::vector<GridMode> gm;
  for (int k = 0; k < n; ++k) {
    const JMode& m = ms[size_t(k)];
    const int64_t t = k == a ? Ta : (k == b ? Tb : 1);
    if (t == m.e) continue;
    gm.push_back({{m.e / t, m.s * t, m.d * t}, tdim[size_t(k)], t});
    if (!al(m.s * t) || !al(m.d * t)) return ch;
  }
  if (gm.size() > size_t(kMaxModes)) return ch;
  std::sort(gm.begin(), gm.end(), [](const GridMode& x, const GridMode& y) {
    return mode_before(x.m, y.m);
  });
  std::vector<JMode> grid;
  for (const GridMode& g : gm) grid.push_back(g.m);
  if (prod_e(grid) >= (int64_t(1) << 32)) return ch;
  const int64_t s_reach = add_chk(mul_chk(mul_chk(Tb - 1, mb.s), eb), seg_bytes);
  const int64_t d_reach = add_chk(mul_chk(mul_chk(Ta - 1, ma.d), eb), Tb * eb);
  if (s_reach >= (int64_t(1) << 31) || d_reach >= (int64_t(1) << 31))
    return ch;

  // tensor-map loads: one box per tile, for sources whose modes a tensor
  // map can describe (at most 5, byte strides multiples of 16 below 2^40,
  // boxes of at most 256 per dimension)
  bool tma = tma_enabled() && !ssb.on() && n <= 5 && Ta <= 256 && Tb <= 256;
  for (int k = 0; k < n && tma; ++k) {
    const JMode& m = ms[size_t(k)];
    if (m.e >= (int64_t(1) << 31)) tma = false;
    if (k != a && (!al(m.s) || m.s * eb >= (int64_t(1) << 40) || m.s <= 0))
      tma = false;
  }
  const bool bulk = tma || (bulk_enabled() && !ssb.on() && Tb <= 128 &&
                            seg_bytes >= kBulkMinSegment);
  // without a swizzle (bulk copies write rows linearly) run the micro-tile
  // index along a first: 8 lanes then read 8 consecutive chunks of a row
  // (LM_TMA_ACFAST=0 keeps the b-first order on tensor-map tiles: stores
  // coalesced, shared reads conflicting)
  // Tensor-map boxes of 128-byte rows with the hardware's 128-byte swizzle
  // (16-byte chunk c of row y at chunk c ^ (y % 8), the tile's width in
  // column regions of Tb rows each): with micro-tiles in warp blocks of 8
  // along b by 4 along a, each quarter-warp reads 8 distinct bank groups and
  // each store instruction writes whole 128-byte lines.  4- and 8-byte
  // elements (R = 4 or 2).
  const bool tma_swz = tma && R == V && (R == 4 || R == 2) &&
                       seg_bytes % 128 == 0 && Tb % 8 == 0 && n_bc % 8 == 0 &&
                       n_ac % 4 == 0 && env_int("LM_TMA_SWIZZLE", 1) != 0;
  const bool acfast = !tma_swz && bulk && n_ac >= 8 &&
                      !(tma && env_int("LM_TMA_ACFAST", 1) == 0);
  const int64_t region = Tb * 128;
  auto block_coords = [&](int64_t j, int64_t* ac, int64_t* bc) {
    const int64_t w = j >> 5, l = j & 31, nwb = n_bc / 8;
    if (R == 4) {
      *bc = 8 * (w % nwb) + 2 * (l >> 3) + (l & 1);
      *ac = 4 * (w / nwb) + ((l >> 1) & 3);
    } else {
      *bc = 8 * (w % nwb) + 4 * ((l >> 3) & 1) + (l & 3);
      *ac = 4 * (w / nwb) + 2 * (l >> 4) + ((l >> 2) & 1);
    }
  };
  const Swz swz128{3, 4, 3};
  auto read_addr = [&](int64_t j, int r, int64_t pitch) {
    if (tma_swz) {
      int64_t ac, bc;
      block_coords(j, &ac, &bc);
      const int64_t lin = (ac >> 3) * region + (ac & 7) * 16 + (bc * R + r) * 128;
      return swz128.apply(lin);
    }
    const int64_t bc = acfast ? j / n_ac : j % n_bc;
    const int64_t ac = acfast ? j % n_ac : j / n_bc;
    return (bc * R + r) * pitch + ac * 16;
  };
  // a tensor-map box lands densely: rows at their own length, no pad
  const SmemLayout best = search_smem(int(threads), Tb, seg_bytes, n_micro,
                                      int(R), 16, read_addr, !bulk, !tma);
  if (best.cost < 0) return ch;

  StagedArgs& A = pc.st;
  A = StagedArgs{};
  fill_grid(A, grid, s_base, d_base, eb, ssb, dsb);
  const int64_t pitch = seg_bytes + best.pad;
  A.n_lchunks = uint32_t(Tb * cps);
  A.cps = uint32_t(cps);
  A.cps_div = make_fastdiv(uint32_t(cps));
  A.nso = 1;
  A.so_ext[0] = uint32_t(Tb);
  A.so_div[0] = make_fastdiv(uint32_t(Tb));
  A.so_s[0] = mul_chk(mb.s, eb);
  A.so_m[0] = uint32_t(pitch);
  A.store_mode = 1;
  A.xr = int32_t(R);
  A.n_micro = uint32_t(n_micro);
  A.n_bc = uint32_t(n_bc);
  A.bc_div = make_fastdiv(uint32_t(n_bc));
  A.n_ac = uint32_t(n_ac);
  A.ac_div = make_fastdiv(uint32_t(n_ac));
  A.x_acfast = acfast ? 1 : 0;
  A.x_pitch = uint32_t(pitch);
  A.x_da = mul_chk(V * ma.d, eb);
  A.x_db = R * eb;
  A.x_vstep = R == V ? mul_chk(ma.d, eb) : 16;
  if (A.x_vstep * R >= (int64_t(1) << 31)) return ch;  // kept in 32 bits
  A.stage_bytes = uint32_t(best.bytes);
  A.m_swz = best.z;
  A.threads = int32_t(threads);
  A.stages = staged_stages();
  A.load_reach = load_reach(A, seg_bytes);
  if (bulk) {
    A.bulk = 1;
    A.bulk_stages = bulk_stages();
    A.n_seg = uint32_t(Tb);
    A.seg_bytes = uint32_t(seg_bytes);
    A.src_reach = src_reach(A);
  }
  if (tma) {
    A.tma = 1;
    A.bulk_stages = tma_stages();
    // tensor copies land on 128-byte boundaries (swizzled ones on 1024):
    // every stage starts on one
    A.stage_bytes = (A.stage_bytes + 1023u) & ~1023u;
    A.t_rank = int32_t(n);
    for (int k = 0; k < n; ++k) {
      const int d = tdim[size_t(k)];
      A.t_dim[d] = uint64_t(ms[size_t(k)].e);
      A.t_stride[d] = uint64_t(mul_chk(ms[size_t(k)].s, eb));
      A.t_box[d] = uint32_t(k == a ? Ta : (k == b ? Tb : 1));
    }
    for (size_t k = 0; k < gm.size(); ++k) {
      A.g_tdim[k] = int32_t(gm[k].tdim);
      A.g_tstep[k] = uint32_t(gm[k].tstep);
    }
    if (tma_swz) {
      A.t_swz128 = 1;
      A.t_regions = uint32_t(seg_bytes / 128);
      A.t_box[0] = uint32_t(128 / eb);
      A.x_blocks = 1;
      A.x_region = uint32_t(region);
      A.x_pitch = 128;
      A.m_swz = swz128;
    }
  }
  pc.path = PATH_STAGED;
  pc.xr = int(R);
  pc.tile_elems = Ta * Tb;
  pc.bank_cost = best.cost;
  pc.bank_ideal = best.ideal;
  pc.bank_read = best.read_cost;
  pc.bank_read_ideal = best.read_ideal;
  ch.ok = true;
  return ch;
}

// Bytes past a tile's origin that its loads reach (one past the last byte).
// Try to plan `ms` (a box of the joint domain) on the STAGED path.  Fills
// pc on success.  May instead request a split of a mode whose extent has no
// good tile divisor.
static StagedChoice plan_staged(const std::vector<JMode>& ms, int64_t s_base,
                                int64_t d_base, const lm_plan& P, Piece& pc) {
  StagedChoice ch;
  const int eb = P.eb;
  const int64_t V = 16 / eb;  // elements per 16-byte chunk
  const int n = int(ms.size());
  int a = -1, b = -1;
  for (int k = 0; k < n; ++k) {
    if (ms[size_t(k)].s == 1 && a < 0) a = k;
    if (ms[size_t(k)].d == 1 && b < 0) b = k;
  }
  if (a < 0 || b < 0) return ch;
  const Swz ssb = to_bytes(P.s_swz, eb), dsb = to_bytes(P.d_swz, eb);
  if ((ssb.on() && ssb.m < 4) || (dsb.on() && dsb.m < 4)) return ch;

  const int64_t target = tile_bytes_target() / eb;  // elements per tile
  std::vector<int64_t> T(size_t(n), 0);
  auto tile_elems = [&] {
    int64_t p = 1;
    for (int k = 0; k < n; ++k)
      if (T[size_t(k)]) p *= T[size_t(k)];
    return p;
  };
  // choose a tile extent near `want` for mode k, or request a split
  auto choose = [&](int k, int64_t want, int64_t mult) -> bool {
    const int64_t e = ms[size_t(k)].e;
    want = std::max<int64_t>(want, 1);
    if (e <= want) {
      T[size_t(k)] = e;
      return true;
    }
    int64_t t = divisor_at_most(e, want, mult);
    if (t == 0 || t * 2 <= want) {
      // no divisor close to `want`: split off the ragged tail of the mode
      int64_t w = std::max<int64_t>(mult, (want / mult) * mult);
      if (e / w >= 1 && e % w) {
        ch.split_mode = k;
        ch.split_at = e - e % w;
        return false;
      }
      t = divisor_at_most(e, want, 1);
    }
    T[size_t(k)] = t;
    return true;
  };

  // 1) destination run: about 128 bytes along the dst-fastest modes
  {
    int cur = b;
    int64_t span = 1;
    const int64_t want = std::max<int64_t>(V, 128 / eb);
    if (!choose(cur, want, V > 1 ? std::min<int64_t>(V, ms[size_t(cur)].e) : 1))
      return ch;
    span = T[size_t(cur)];
    while (T[size_t(cur)] == ms[size_t(cur)].e && span < want) {
      int nxt = -1;
      for (int k = 0; k < n; ++k)
        if (!T[size_t(k)] && ms[size_t(k)].d == span) nxt = k;
      if (nxt < 0) break;
      if (!choose(nxt, (want + span - 1) / span, 1)) return ch;
      span *= T[size_t(nxt)];
      cur = nxt;
    }
  }
  // 2) source run: the src-fastest mode, sized to fill the tile target
  if (!T[size_t(a)]) {
    const int64_t want =
        std::max<int64_t>(128 / eb, target / std::max<int64_t>(tile_elems(), 1));
    if (!choose(a, want, std::min<int64_t>(V, ms[size_t(a)].e))) return ch;
  }
  // 3) grow until the tile holds about `target` elements: first along the
  //    destination's contiguous chain, then the partial src/dst modes, then a
  //    new outer mode
  for (int guard = 0; guard < 64 && tile_elems() * 2 <= target; ++guard) {
    // dst chain continuation
    int64_t span = 1;
    int cur = b;
    std::vector<bool> in_chain(size_t(n), false);
    for (;;) {
      in_chain[size_t(cur)] = true;
      span *= T[size_t(cur)];
      if (T[size_t(cur)] != ms[size_t(cur)].e) break;
      int nxt = -1;
      for (int k = 0; k < n; ++k)
        if (!in_chain[size_t(k)] && ms[size_t(k)].d == span) nxt = k;
      if (nxt < 0 || !T[size_t(nxt)]) {
        if (nxt >= 0) {
          if (!choose(nxt, std::max<int64_t>(1, target / tile_elems()), 1))
            return ch;
          cur = -1;
        }
        break;
      }
      cur = nxt;
    }
    if (cur == -1) continue;
    // partial modes: double the src-fast one, then the dst-fast one
    bool grown = false;
    for (int k : {a, b}) {
      const int64_t e = ms[size_t(k)].e, t = T[size_t(k)];
      if (t < e && e % (2 * t) == 0 && tile_elems() * 2 <= target) {
        T[size_t(k)] = 2 * t;
        grown = true;
        break;
      }
    }
    if (grown) continue;
    // a new outer mode
    int best = -1;
    for (int k = 0; k < n; ++k) {
      if (T[size_t(k)]) continue;
      if (best < 0 || std::min(ms[size_t(k)].s, ms[size_t(k)].d) <
                          std::min(ms[size_t(best)].s, ms[size_t(best)].d))
        best = k;
    }
    if (best < 0) break;
    if (!choose(best, std::max<int64_t>(1, target / tile_elems()), 1))
      return ch;
  }

  // ---- chains over the final tile ---------------------------------------
  std::vector<int> tile_modes;
  for (int k = 0; k < n; ++k)
    if (T[size_t(k)]) tile_modes.push_back(k);
  if (tile_modes.size() > size_t(kMaxTile)) return ch;

  // src chain: from a, the tile mode with the smallest stride at or beyond
  // the current span, gaps of at most one chunk, through full modes only
  std::vector<int> s_chain{a};
  int64_t s_span = T[size_t(a)];
  {
    std::vector<bool> used(size_t(n), false);
    used[size_t(a)] = true;
    int cur = a;
    while (T[size_t(cur)] == ms[size_t(cur)].e) {
      int nxt = -1;
      for (int k : tile_modes) {
        if (used[size_t(k)] || ms[size_t(k)].s < s_span) continue;
        if ((ms[size_t(k)].s - s_span) * eb > 16) continue;
        if (nxt < 0 || ms[size_t(k)].s < ms[size_t(nxt)].s) nxt = k;
      }
      if (nxt < 0) break;
      used[size_t(nxt)] = true;
      s_span = ms[size_t(nxt)].s * (T[size_t(nxt)] - 1) + s_span;
      s_chain.push_back(nxt);
      cur = nxt;
    }
  }
  // dst chain: exact contiguity
  std::vector<int> d_chain{b};
  int64_t d_span = T[size_t(b)];
  {
    std::vector<bool> used(size_t(n), false);
    used[size_t(b)] = true;
    int cur = b;
    while (T[size_t(cur)] == ms[size_t(cur)].e) {
      int nxt = -1;
      for (int k : tile_modes)
        if (!used[size_t(k)] && ms[size_t(k)].d == d_span) nxt = k;
      if (nxt < 0) break;
      used[size_t(nxt)] = true;
      d_span *= T[size_t(nxt)];
      d_chain.push_back(nxt);
      cur = nxt;
    }
  }
  auto in = [](const std::vector<int>& v, int k) {
    return std::find(v.begin(), v.end(), k) != v.end();
  };
  std::vector<int> s_outer, d_outer;
  for (int k : tile_modes) {
    if (!in(s_chain, k)) s_outer.push_back(k);
    if (!in(d_chain, k)) d_outer.push_back(k);
  }
  if (s_outer.size() > size_t(kMaxTile) || d_outer.size() > size_t(kMaxTile) ||
      d_chain.size() > size_t(kMaxTile))
    return ch;

  // ---- alignment: every chunk start 16-byte aligned ----------------------
  const int64_t seg_bytes = ((s_span * eb + 15) / 16) * 16;
  {
    // the kernel keeps offsets inside a tile in 32 bits
    int64_t s_reach = seg_bytes, d_reach = 16;
    for (int k : tile_modes) {
      s_reach = add_chk(s_reach, mul_chk(mul_chk(T[size_t(k)] - 1, ms[size_t(k)].s), eb));
      d_reach = add_chk(d_reach, mul_chk(mul_chk(T[size_t(k)] - 1, ms[size_t(k)].d), eb));
    }
    if (s_reach >= (int64_t(1) << 31) || d_reach >= (int64_t(1) << 31)) return ch;
  }
  if ((d_span * eb) % 16) return ch;
  auto al = [&](int64_t elems) { return (elems * eb) % 16 == 0; };
  if (!al(s_base) || !al(d_base)) return ch;
  for (int k : s_outer)
    if (!al(ms[size_t(k)].s)) return ch;
  for (int k : d_outer)
    if (!al(ms[size_t(k)].d)) return ch;
  std::vector<JMode> grid;
  for (int k = 0; k < n; ++k) {
    const JMode& m = ms[size_t(k)];
    const int64_t t = T[size_t(k)] ? T[size_t(k)] : 1;
    if (t == m.e) continue;
    grid.push_back({m.e / t, m.s * t, m.d * t});
    if (!al(m.s * t) || !al(m.d * t)) return ch;
  }
  if (grid.size() > size_t(kMaxModes)) return ch;
  std::sort(grid.begin(), grid.end(), mode_before);
  const int64_t n_tiles = prod_e(grid);
  if (n_tiles >= (int64_t(1) << 32)) return ch;

  // ---- shared-memory layout: segment pitch and XOR swizzle ---------------
  int64_t n_seg = 1;
  for (int k : s_outer) n_seg *= T[size_t(k)];
  const int64_t cps = seg_bytes / 16;
  const int64_t n_l = n_seg * cps;
  const int64_t n_s = tile_elems() / V;
  const int64_t cpd = d_span * eb / 16;
  // (these limits match GatherStore: load chunks and store chunks per thread)
  const int max_s = std::max(1, std::min(4, 16 / int(V)));
  const int max_l = eb >= 8 ? 8 : 4;
  if (n_l > kThreads * max_l || n_s > int64_t(kThreads) * max_s) return ch;

  // smem bytes per coordinate of each tile mode for a given pitch
  auto smem_m = [&](int64_t pitch, std::vector<int64_t>& m) {
    m.assign(size_t(n), 0);
    for (int k : s_chain) m[size_t(k)] = ms[size_t(k)].s * eb;
    int64_t w = pitch;
    for (int k : s_outer) {
      m[size_t(k)] = w;
      w *= T[size_t(k)];
    }
  };
  // linear smem address of element e of store chunk j
  int64_t cached_pitch = -1;
  std::vector<int64_t> mcache;
  auto gather_addr = [&](int64_t j, int e, int64_t pitch) {
    if (pitch != cached_pitch) {
      smem_m(pitch, mcache);
      cached_pitch = pitch;
    }
    int64_t o = j / cpd, p = j % cpd, addr = 0;
    for (int k : d_outer) {
      addr += (o % T[size_t(k)]) * mcache[size_t(k)];
      o /= T[size_t(k)];
    }
    int64_t q = p * V + e;
    for (int k : d_chain) {
      addr += (q % T[size_t(k)]) * mcache[size_t(k)];
      q /= T[size_t(k)];
    }
    return addr;
  };
  const bool bulk = bulk_enabled() && !ssb.on() && n_seg <= 128 &&
                    seg_bytes >= kBulkMinSegment;
  const SmemLayout best = search_smem(kThreads, n_seg, seg_bytes, n_s,
                                      int(V), eb, gather_addr, !bulk);
  if (best.cost < 0) return ch;

  // ---- fill the kernel arguments -----------------------------------------
  StagedArgs& A = pc.st;
  A = StagedArgs{};
  const int64_t pitch = seg_bytes + best.pad;
  std::vector<int64_t> m;
  smem_m(pitch, m);
  fill_grid(A, grid, s_base, d_base, eb, ssb, dsb);
  A.n_lchunks = uint32_t(n_l);
  A.cps = uint32_t(cps);
  A.cps_div = make_fastdiv(uint32_t(cps));
  A.nso = int32_t(s_outer.size());
  for (size_t i = 0; i < s_outer.size(); ++i) {
    const int k = s_outer[i];
    A.so_ext[i] = uint32_t(T[size_t(k)]);
    A.so_div[i] = make_fastdiv(uint32_t(T[size_t(k)]));
    A.so_s[i] = mul_chk(ms[size_t(k)].s, eb);
    A.so_m[i] = uint32_t(m[size_t(k)]);
  }
  A.n_schunks = uint32_t(n_s);
  A.cpd = uint32_t(cpd);
  A.cpd_div = make_fastdiv(uint32_t(cpd));
  A.ndo = int32_t(d_outer.size());
  for (size_t i = 0; i < d_outer.size(); ++i) {
    const int k = d_outer[i];
    A.do_ext[i] = uint32_t(T[size_t(k)]);
    A.do_div[i] = make_fastdiv(uint32_t(T[size_t(k)]));
    A.do_d[i] = mul_chk(ms[size_t(k)].d, eb);
    A.do_m[i] = uint32_t(m[size_t(k)]);
  }
  A.ndi = int32_t(d_chain.size());
  for (size_t i = 0; i < d_chain.size(); ++i) {
    const int k = d_chain[i];
    A.di_ext[i] = uint32_t(T[size_t(k)]);
    A.di_div[i] = make_fastdiv(uint32_t(T[size_t(k)]));
    A.di_m[i] = uint32_t(m[size_t(k)]);
  }
  A.stage_bytes = uint32_t(best.bytes);
  A.m_swz = best.z;
  A.store_mode = 0;
  A.threads = kThreads;
  A.stages = staged_stages();
  A.load_reach = load_reach(A, seg_bytes);
  if (bulk) {
    A.bulk = 1;
    A.bulk_stages = bulk_stages();
    A.n_seg = uint32_t(n_seg);
    A.seg_bytes = uint32_t(seg_bytes);
    A.src_reach = src_reach(A);
  }
  pc.path = PATH_STAGED;
  pc.tile_elems = tile_elems();
  pc.bank_cost = best.cost;
  pc.bank_ideal = best.ideal;
  pc.bank_read = best.read_cost;
  pc.bank_read_ideal = best.read_ideal;
  ch.ok = true;
  return ch;
}

// VEC when a unit-stride run shared by both sides gives 16-byte vectors (or
// narrower vectors when `allow_narrow`).  May request a split of the run.
static StagedChoice plan_vec(const std::vector<JMode>& ms, int64_t s_base,
                             int64_t d_base, const lm_plan& P, Piece& pc,
                             bool allow_narrow) {
  StagedChoice ch;
  const int eb = P.eb;
  int r = -1;
  for (size_t k = 0; k < ms.size(); ++k)
    if (ms[k].s == 1 && ms[k].d == 1) r = int(k);
  if (r < 0) return ch;
  auto fits = [&](int64_t V, bool check_run) {
    if (check_run && ms[size_t(r)].e % V) return false;
    for (size_t k = 0; k < ms.size(); ++k) {
      if (int(k) == r) continue;
      if (ms[k].s % V || ms[k].d % V) return false;
    }
    if (s_base % V || d_base % V) return false;
    if (P.s_swz.on() && (int64_t(1) << P.s_swz.m) < V) return false;
    if (P.d_swz.on() && (int64_t(1) << P.d_swz.m) < V) return false;
    return true;
  };
  const int64_t vmax = 16 / eb;
  const int64_t e = ms[size_t(r)].e;
  if (vmax > 1 && e % vmax && e >= 2 * vmax && fits(vmax, false)) {
    ch.split_mode = r;
    ch.split_at = e - e % vmax;
    return ch;
  }
  int64_t V = vmax;
  while (V > 1 && !fits(V, true)) V /= 2;
  const int vb = int(V * eb);
  if (vb < 16 && !allow_narrow) return ch;
  if (vb < 4) return ch;
  std::vector<JMode> rest;
  for (size_t k = 0; k < ms.size(); ++k)
    if (int(k) != r) rest.push_back(ms[k]);
  std::sort(rest.begin(), rest.end(), mode_before);
  if (rest.size() + 1 > size_t(kMaxModes)) return ch;
  VecArgs& A = pc.vec;
  A = VecArgs{};
  const int64_t nvec = prod_e(ms) / V;
  if (nvec >= (int64_t(1) << 32)) return ch;
  A.n_vec = uint32_t(nvec);
  A.nm = int32_t(rest.size() + 1);
  A.ext[0] = uint32_t(e / V);
  A.div[0] = make_fastdiv(A.ext[0]);
  A.s[0] = V * eb;
  A.d[0] = V * eb;
  for (size_t k = 0; k < rest.size(); ++k) {
    A.ext[k + 1] = uint32_t(rest[k].e);
    A.div[k + 1] = make_fastdiv(uint32_t(rest[k].e));
    A.s[k + 1] = mul_chk(rest[k].s, eb);
    A.d[k + 1] = mul_chk(rest[k].d, eb);
  }
  A.s_base = mul_chk(s_base, eb);
  A.d_base = mul_chk(d_base, eb);
  A.s_swz = to_bytes(P.s_swz, eb);
  A.d_swz = to_bytes(P.d_swz, eb);
  // tiled form: about 1024 vectors per tile over the leading modes, so each
  // thread's offsets inside a tile are computed once
  {
    std::vector<JMode> vm;  // vector units: the run first, then the rest
    vm.push_back({e / V, V, V});
    for (const JMode& m : rest) vm.push_back(m);
    const int64_t want = 256 * vec_unroll();
    int64_t tile = 1;
    std::vector<int64_t> T;
    for (size_t k = 0; k < vm.size(); ++k) {
      if (tile * vm[k].e <= want) {
        T.push_back(vm[k].e);
        tile *= vm[k].e;
        continue;
      }
      const int64_t t = divisor_at_most(vm[k].e, want / tile, 1);
      T.push_back(t);
      tile *= t;
      break;
    }
    int64_t s_reach = vb, d_reach = vb;
    for (size_t k = 0; k < T.size(); ++k) {
      s_reach = add_chk(s_reach, mul_chk(mul_chk(T[k] - 1, vm[k].s), eb));
      d_reach = add_chk(d_reach, mul_chk(mul_chk(T[k] - 1, vm[k].d), eb));
    }
    std::vector<JMode> grid;
    for (size_t k = 0; k < vm.size(); ++k) {
      const int64_t t = k < T.size() ? T[k] : 1;
      if (t != vm[k].e) grid.push_back({vm[k].e / t, vm[k].s * t, vm[k].d * t});
    }
    if (tile >= 256 && s_reach < (int64_t(1) << 31) &&
        d_reach < (int64_t(1) << 31) && grid.size() <= size_t(kMaxModes) &&
        prod_e(grid) < (int64_t(1) << 32)) {
      A.tiled = 1;
      A.unroll = vec_unroll();
      A.tile_vecs = uint32_t(tile);
      A.nt = int32_t(T.size());
      for (size_t k = 0; k < T.size(); ++k) {
        A.t_ext[k] = uint32_t(T[k]);
        A.t_div[k] = make_fastdiv(uint32_t(T[k]));
        A.t_s[k] = mul_chk(vm[k].s, eb);
        A.t_d[k] = mul_chk(vm[k].d, eb);
      }
      A.n_tiles = uint32_t(prod_e(grid));
      A.ng = int32_t(grid.size());
      uint32_t pre = 1;
      for (size_t k = 0; k < grid.size(); ++k) {
        A.g_ext[k] = uint32_t(grid[k].e);
        A.g_pre[k] = make_fastdiv(pre);
        A.g_div[k] = make_fastdiv(uint32_t(grid[k].e));
        A.g_s[k] = mul_chk(grid[k].s, eb);
        A.g_d[k] = mul_chk(grid[k].d, eb);
        pre *= uint32_t(grid[k].e);
      }
    }
  }
  pc.path = PATH_VEC;
  pc.vec_bytes = vb;
  ch.ok = true;
  return ch;
}

static void plan_box(lm_plan& P, std::vector<JMode> ms, int64_t s_base,
                     int64_t d_base, int depth) {
  ms = coalesce_joint(ms);
  const int64_t size = prod_e(ms);
  if (size == 0) return;
  if (depth > 24 || ms.size() > size_t(kMaxModes)) {
    Piece pc;
    pc.modes = ms;
    pc.s_base = s_base;
    pc.d_base = d_base;
    pc.gen = generic_for_modes(ms, s_base, d_base, P);
    P.pieces.push_back(std::move(pc));
    return;
  }
  auto split = [&](int k, int64_t at) {
    std::vector<JMode> lo = ms, hi = ms;
    lo[size_t(k)].e = at;
    hi[size_t(k)].e = ms[size_t(k)].e - at;
    plan_box(P, lo, s_base, d_base, depth + 1);
    plan_box(P, hi, add_chk(s_base, mul_chk(at, ms[size_t(k)].s)),
             add_chk(d_base, mul_chk(at, ms[size_t(k)].d)), depth + 1);
  };
  if (size >= kMaxPiece) {
    int k = 0;
    for (size_t j = 1; j < ms.size(); ++j)
      if (ms[j].e > ms[size_t(k)].e) k = int(j);
    // halve the longest mode at a multiple of 64 coordinates, so both
    // halves start on 16-byte boundaries whenever the whole did
    int64_t at = ms[size_t(k)].e / 2;
    if (ms[size_t(k)].e >= 256) at = at / 64 * 64;
    split(k, at);
    return;
  }
  Piece pc;
  pc.modes = ms;
  pc.s_base = s_base;
  pc.d_base = d_base;
  pc.gen = generic_for_modes(ms, s_base, d_base, P);
  if (size > kSmall) {
    StagedChoice c = plan_vec(ms, s_base, d_base, P, pc, false);
    if (c.split_mode >= 0) return split(c.split_mode, c.split_at);
    if (!c.ok && !transpose_disabled()) {
      c = plan_transpose(ms, s_base, d_base, P, pc);
      if (c.split_mode >= 0) return split(c.split_mode, c.split_at);
    }
    if (!c.ok) {
      c = plan_staged(ms, s_base, d_base, P, pc);
      if (c.split_mode >= 0) return split(c.split_mode, c.split_at);
    }
    if (!c.ok) c = plan_vec(ms, s_base, d_base, P, pc, true);
    if (!c.ok) pc.path = PATH_GENERIC;
  }
  P.pieces.push_back(std::move(pc));
}

static std::string describe(const lm_plan& P) {
  std::ostringstream os;
  os << "{\"size\":" << P.size << ",\"elem_bytes\":" << P.eb
     << ",\"joint\":" << (P.joint ? "true" : "false")
     << ",\"src_range\":[" << P.src_lo << ',' << P.src_hi
     << "],\"dst_range\":[" << P.dst_lo << ',' << P.dst_hi
     << "],\"dst_own\":" << (P.dst_own ? "true" : "false")
     << ",\"pieces\":[";
  for (size_t i = 0; i < P.pieces.size(); ++i) {
    const Piece& pc = P.pieces[i];
    if (i) os << ',';
    const char* path = pc.path == PATH_VEC      ? "VEC"
                       : pc.path == PATH_STAGED ? "STAGED"
                       : pc.path == PATH_ZIP    ? "ZIP"
                       : pc.path == PATH_GTILE  ? "GTILE"
                                                : "GENERIC";
    os << "{\"path\":\"" << path << "\",\"modes\":[";
    for (size_t k = 0; k < pc.modes.size(); ++k) {
      if (k) os << ',';
      os << '[' << pc.modes[k].e << ',' << pc.modes[k].s << ','
         << pc.modes[k].d << ']';
    }
    os << "],\"s_base\":" << pc.s_base << ",\"d_base\":" << pc.d_base;
    if (!P.joint)
      os << ",\"index_begin\":" << pc.gen.i0 << ",\"index_count\":"
         << pc.gen.n;
    if (pc.path == PATH_VEC)
      os << ",\"vec_bytes\":" << pc.vec_bytes << ",\"tiled\":"
         << (pc.vec.tiled ? "true" : "false") << ",\"tile_vecs\":"
         << pc.vec.tile_vecs << ",\"n_tiles\":" << pc.vec.n_tiles;
    if (pc.path == PATH_ZIP)
      os << ",\"vec_bytes\":16,\"rows\":" << pc.vec.zip_rows
         << ",\"n_vec\":" << pc.vec.n_vec;
    if (pc.path == PATH_GTILE) {
      const GTileArgs& g = pc.gt;
      os << ",\"outer\":\"" << (g.outer_src ? "src" : "dst")
         << "\",\"u_extent\":" << g.W << ",\"v_extent\":" << g.nv
         << ",\"tma\":" << (g.tma ? "true" : "false")
         << ",\"tile\":[" << g.tile_u << ',' << kGtV << "],\"n_tiles\":"
         << uint64_t(g.n_ut) * g.n_vt
         << ",\"offsets32\":" << (g.narrow ? "true" : "false");
      // each part's leaves [extent, byte stride] and the steps its threads
      // take: the step's digits, its offset change without carries and the
      // extra change of a carry out of each leaf
      auto leaves = [&](const char* name, int n, const uint32_t* ext,
                        const int64_t* str) {
        os << ",\"" << name << "_leaves\":[";
        for (int k = 0; k < n; ++k)
          os << (k ? "," : "") << '[' << ext[k] << ',' << str[k] << ']';
        os << ']';
      };
      bool first = true;
      auto step = [&](const char* name, int n, const uint32_t* d,
                      int64_t dsum, const int64_t* cadj) {
        os << (first ? "" : ",") << '"' << name << "\":{\"digits\":[";
        first = false;
        for (int k = 0; k < n; ++k) os << (k ? "," : "") << d[k];
        os << "],\"dstep\":" << dsum << ",\"cadj\":[";
        for (int k = 0; k < n; ++k) os << (k ? "," : "") << cadj[k];
        os << "]}";
      };
      leaves("lo", g.n_lo, g.lo_ext, g.lo_str);
      leaves("hi", g.n_hi, g.hi_ext, g.hi_str);
      leaves("in", g.n_in, g.in_ext, g.in_str);
      os << ",\"steps\":{";
      step("lo", g.n_lo, g.lo_step, g.lo_dstep, g.lo_cadj);
      step("in", g.n_in, g.in_step, g.in_dstep, g.in_cadj);
      if (g.tma) {
        step("in_next_v", g.n_in, g.in_step1, g.in_dstep1, g.in_cadj);
        step("in_next_chunk", g.n_in, g.in_jump, g.in_djump, g.in_cadj);
      }
      os << '}';
    }
    if (pc.path == PATH_STAGED) {
      const StagedArgs& A = pc.st;
      os << ",\"tile_elems\":" << pc.tile_elems << ",\"n_tiles\":" << A.n_tiles
         << ",\"load_chunks\":" << A.n_lchunks
         << ",\"store_chunks\":" << A.n_schunks
         << ",\"store\":\"" << (A.store_mode ? "transpose" : "gather")
         << "\",\"rows\":" << A.xr << ",\"threads\":" << A.threads
         << ",\"stages\":" << (A.bulk ? A.bulk_stages : A.stages)
         << ",\"bulk\":"
         << (A.bulk ? "true" : "false") << ",\"tma\":"
         << (A.tma ? "true" : "false") << ",\"tma_swizzle\":"
         << (A.t_swz128 ? "true" : "false")
         << ",\"stage_bytes\":" << A.stage_bytes << ",\"smem_swizzle\":["
         << A.m_swz.b << ',' << A.m_swz.m << ',' << A.m_swz.s << ']'
         << ",\"bank_wavefronts\":" << pc.bank_cost
         << ",\"bank_wavefronts_ideal\":" << pc.bank_ideal
         << ",\"bank_read_wavefronts\":" << pc.bank_read
         << ",\"bank_read_wavefronts_ideal\":" << pc.bank_read_ideal;
    }
    os << '}';
  }
  os << "]}";
  return os.str();
}

}  // namespace lm

using lm::fail;

namespace lm {

// The search behind lm_stripmined_tune.  With `partition`, only maps whose
// one Pitch x Strips group holds every thread (P*S == threads) and whose P
// and S divide the tile's vectors per row and rows are candidates: those
// are the pitch-linear thread layouts (P, S):(1, P) that tile the tile, the
// form a local_partition thread layout can take.
int stripmined_search(int64_t threads, int64_t k_row, int64_t rows,
                      int64_t ld, int elem_bytes, int vec_elems,
                      const lm_layout* smem, bool partition, int64_t* pitch,
                      int64_t* strips, int64_t* segments,
                      int64_t* wavefronts) {
  if (threads < 1 || threads > 1024 || k_row < 1 || rows < 1 || ld < k_row ||
      vec_elems < 1 || k_row % vec_elems)
    return LM_E_INVALID;
  const int64_t vb = int64_t(elem_bytes) * vec_elems;
  if (elem_bytes < 1 || vb > 16 || (vb & (vb - 1)) ||
      (elem_bytes & (elem_bytes - 1)))
    return LM_E_INVALID;
  if (smem) {
    const std::vector<Node> m = top_modes(*smem);
    if (m.size() != 2) return LM_E_INVALID;
    int64_t s0 = 1, s1 = 1;
    for (const Leaf& l : flatten(m[0])) s0 *= l.e;
    for (const Leaf& l : flatten(m[1])) s1 *= l.e;
    if (s0 != rows || s1 != k_row) return LM_E_INVALID;
  }
  try {
    const int64_t R = k_row / vec_elems;  // vectors per row
    int64_t best_p = 0, best_s = 0, best_seg = -1, best_wf = -1;
    std::vector<int64_t> gaddr(32), saddr(32);
    bool valid[32];
    for (int64_t P = 1; P <= R && P <= threads; P *= 2)
      for (int64_t S = 1; S <= rows && P * S <= threads; S *= 2) {
        if (partition && (P * S != threads || R % P || rows % S)) continue;
        int64_t seg = 0, wf = 0;
        bool fits = true;
        for (int64_t w0 = 0; w0 < threads && fits; w0 += 32) {
          int64_t segs[32];
          int ns = 0;
          for (int l = 0; l < 32; ++l) {
            const int64_t t = w0 + l;
            valid[l] = t < threads;
            gaddr[size_t(l)] = saddr[size_t(l)] = 0;
            if (!valid[l]) continue;
            const int64_t d = t / P;
            const int64_t row = d % S + (d / S) * P * S;
            const int64_t col = (t % P) * vec_elems;
            if (row >= rows) {
              fits = false;
              break;
            }
            const int64_t g = mul_chk(row * ld + col, elem_bytes) / 128;
            bool seen = false;
            for (int q = 0; q < ns; ++q) seen = seen || segs[q] == g;
            if (!seen) segs[ns++] = g;
            const int64_t o =
                smem ? smem->swz.apply(eval_affine(smem->leaves,
                                                   row + rows * col))
                     : row * k_row + col;
            saddr[size_t(l)] = mul_chk(o, elem_bytes);
            if (saddr[size_t(l)] % vb) return LM_E_INVALID;
          }
          if (!fits) break;
          seg += ns;
          wf += warp_wavefronts(saddr.data(), valid, int(vb));
        }
        if (!fits) continue;
        const bool better =
            best_seg < 0 || seg < best_seg ||
            (seg == best_seg &&
             (wf < best_wf || (wf == best_wf && (P > best_p ||
                                                 (P == best_p && S > best_s)))));
        if (better) {
          best_p = P;
          best_s = S;
          best_seg = seg;
          best_wf = wf;
        }
      }
    if (best_seg < 0) return LM_E_NOT_REPRESENTABLE;
    *pitch = best_p;
    *strips = best_s;
    *segments = best_seg;
    *wavefronts = best_wf;
    return LM_OK;
  } catch (const Error& e) {
    return e.status;
  }
}

}  // namespace lm

extern "C" {

// Shared-memory wavefronts of the accesses `access` describes: access i
// (colex over its domain) is lane i % 32 of warp access i / 32 and reads
// access_bytes at byte address access(i) * elem_bytes.  Same bank model as
// the planner's layout search (32 banks of 4 bytes; 16-byte accesses served
// 8 lanes at a time, 8-byte ones 16 at a time; one word read by several
// lanes is a broadcast).
int lm_smem_wavefronts(const lm_layout* access, int elem_bytes,
                       int access_bytes, int64_t* wavefronts, int64_t* ideal) {
  auto pow2_le16 = [](int v) { return v >= 1 && v <= 16 && !(v & (v - 1)); };
  if (!access || !wavefronts || !ideal || !pow2_le16(elem_bytes) ||
      !pow2_le16(access_bytes))
    return LM_E_INVALID;
  if (access->size > (int64_t(1) << 24)) return LM_E_INVALID;
  try {
    int64_t total = 0, best = 0;
    std::vector<int64_t> addr(32);
    bool valid[32];
    for (int64_t w0 = 0; w0 < access->size; w0 += 32) {
      int cnt = 0;
      for (int l = 0; l < 32; ++l) {
        const int64_t i = w0 + l;
        valid[l] = i < access->size;
        addr[size_t(l)] = 0;
        if (!valid[l]) continue;
        ++cnt;
        const int64_t off = access->swz.apply(
            lm::eval_affine(access->leaves, i));
        const int64_t a = lm::mul_chk(off, elem_bytes);
        if (a < 0 || a % access_bytes) return LM_E_INVALID;
        addr[size_t(l)] = a;
      }
      total += lm::wavefronts(addr.data(), valid, 32, access_bytes);
      // per phase: its lanes' bytes over 128, at least one
      const int per_phase = access_bytes <= 4 ? 32 : 128 / access_bytes;
      for (int p0 = 0; p0 < cnt; p0 += per_phase) {
        const int n = std::min(cnt - p0, per_phase);
        best += std::max<int64_t>(1, (int64_t(n) * access_bytes + 127) / 128);
      }
    }
    *wavefronts = total;
    *ideal = best;
    return LM_OK;
  } catch (const lm::Error& e) {
    return e.status;
  } catch (const std::bad_alloc&) {
    return LM_E_NOMEM;
  }
}

// Pitch and Strips of the stripmined thread map for one pass of `threads`
// vector accesses over a tile, chosen by the cost of that pass: the
// 128-byte global segments every warp touches, then its shared-memory
// wavefronts under the bank model, then the larger Pitch and Strips.
int lm_stripmined_tune(int64_t threads, int64_t k_row, int64_t rows,
                       int64_t ld, int elem_bytes, int vec_elems,
                       const lm_layout* smem, int64_t* pitch, int64_t* strips,
                       int64_t* segments, int64_t* wavefronts) {
  if (!pitch || !strips || !segments || !wavefronts) return LM_E_INVALID;
  return lm::stripmined_search(threads, k_row, rows, ld, elem_bytes,
                               vec_elems, smem, false, pitch, strips,
                               segments, wavefronts);
}

}  // extern "C"

namespace lm {

// Plan shard `rank` of `world` of the copy (world == 1: the whole copy).
// Joint plans split the joint mode with the largest destination stride
// among those with at least `world` coordinates into `world` balanced
// ranges; other pairs split the logical index range.
static int plan_copy_impl(const lm_layout* src, const lm_layout* dst,
                          int elem_bytes, int rank, int world, lm_plan** out) {
  if (out) *out = nullptr;
  try {
    if (!src || !dst || !out || world < 1 || rank < 0 || rank >= world)
      fail(LM_E_INVALID);
    if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 &&
        elem_bytes != 8 && elem_bytes != 16)
      fail(LM_E_INVALID);
    if (src->size != dst->size) fail(LM_E_INCOMPATIBLE);
    auto P = std::make_unique<lm_plan>();
    P->eb = elem_bytes;
    P->size = src->size;
    P->src_cosize = src->cosize;
    P->dst_cosize = dst->cosize;
    P->s_swz = src->swz;
    P->d_swz = dst->swz;
    // byte offsets must fit int64
    mul_chk(std::max(P->src_cosize, P->dst_cosize), elem_bytes);
    bool dst_own = false;
    if (P->size > 0) {
      if (!affine_injective(dst->leaves)) fail(LM_E_NOT_INJECTIVE);
      std::vector<JMode> jm;
      if (refine_sides(src->leaves, dst->leaves, jm)) {
        P->joint = true;
        jm = coalesce_joint(jm);
        int64_t s_base = 0, d_base = 0;
        if (world > 1 && !jm.empty()) {
          // the largest-stride mode that has at least `world` coordinates,
          // else the longest mode
          size_t k = jm.size();
          for (size_t j = 0; j < jm.size(); ++j)
            if (jm[j].e >= world && (k == jm.size() || jm[j].d > jm[k].d))
              k = j;
          if (k == jm.size()) {
            k = 0;
            for (size_t j = 1; j < jm.size(); ++j)
              if (jm[j].e > jm[k].e) k = j;
          }
          const int64_t e = jm[k].e;
          const int64_t lo = e * rank / world, hi = e * (rank + 1) / world;
          s_base = mul_chk(lo, jm[k].s);
          d_base = mul_chk(lo, jm[k].d);
          // the shard owns [lo*D, hi*D) of the destination when every
          // other mode fits inside one step D of the split mode and the
          // boundaries fall on whole 16-byte chunks and swizzle blocks
          int64_t span = 1;
          for (size_t j = 0; j < jm.size(); ++j)
            if (j != k) span = add_chk(span, mul_chk(jm[j].e - 1, jm[j].d));
          int64_t blk = std::max<int64_t>(1, 16 / elem_bytes);
          if (P->d_swz.on())
            blk = std::max(blk, int64_t(1) << (P->d_swz.b + P->d_swz.m +
                                               P->d_swz.s));
          const int64_t D = jm[k].d;
          dst_own = span <= D && mul_chk(lo, D) % blk == 0 &&
                    (hi == e || mul_chk(hi, D) % blk == 0);
          jm[k].e = hi - lo;
        }
        plan_box(*P, jm, s_base, d_base, 0);
      } else {
        P->joint = false;
        const int64_t lo = P->size * rank / world;
        const int64_t hi = P->size * (rank + 1) / world;
        if (hi > lo) {
          Piece pc;
          pc.path = PATH_GENERIC;
          std::vector<Leaf> sl = coalesce_leaves(src->leaves);
          std::vector<Leaf> dl = coalesce_leaves(dst->leaves);
          pc.gen = make_generic(sl, dl, hi - lo, 0, 0, P->s_swz, P->d_swz,
                                elem_bytes);
          pc.gen.i0 = uint64_t(lo);
          if (uint64_t(hi) >= (uint64_t(1) << 31)) pc.gen.wide = 1;
          if (world == 1 && plan_gtile(sl, dl, P->size, P->s_swz, P->d_swz,
                                       elem_bytes, pc.gt))
            pc.path = PATH_GTILE;
          P->pieces.push_back(std::move(pc));
        }
      }
    }
    P->src_lo = P->dst_lo = 0;
    P->src_hi = P->src_cosize;
    P->dst_hi = P->dst_cosize;
    P->dst_own = world == 1 || dst_own;
    if (P->joint && world > 1) {
      // the offsets the pieces reach, widened to whole swizzle blocks and
      // to 16-byte chunks (the loads move whole chunks)
      int64_t slo = P->src_cosize, shi = 0, dlo = P->dst_cosize, dhi = 0;
      for (const Piece& pc : P->pieces) {
        int64_t sa = pc.s_base, sb = pc.s_base, da = pc.d_base, db = pc.d_base;
        for (const JMode& m : pc.modes) {
          sb = add_chk(sb, mul_chk(m.e - 1, m.s));
          db = add_chk(db, mul_chk(m.e - 1, m.d));
        }
        slo = std::min(slo, sa);
        shi = std::max(shi, sb + 1);
        dlo = std::min(dlo, da);
        dhi = std::max(dhi, db + 1);
      }
      auto widen = [&](int64_t& lo, int64_t& hi, const Swz& z, int64_t cos) {
        int64_t blk = std::max<int64_t>(1, 16 / elem_bytes);
        if (z.on()) blk = std::max(blk, int64_t(1) << (z.b + z.m + z.s));
        lo = lo / blk * blk;
        hi = std::min(cos, (hi + blk - 1) / blk * blk);
        if (lo >= hi) lo = hi = 0;
      };
      if (!P->pieces.empty()) {
        widen(slo, shi, P->s_swz, P->src_cosize);
        widen(dlo, dhi, P->d_swz, P->dst_cosize);
        P->src_lo = slo;
        P->src_hi = shi;
        P->dst_lo = dlo;
        P->dst_hi = dhi;
      } else {
        P->src_hi = P->dst_hi = 0;
      }
    }
    P->describe = describe(*P);
    *out = P.release();
    return LM_OK;
  } catch (const Error& e) {
    return e.status;
  } catch (const std::bad_alloc&) {
    return LM_E_NOMEM;
  } catch (...) {
    return LM_E_INVALID;
  }
}

}  // namespace lm

extern "C" {

int lm_plan_copy(const lm_layout* src, const lm_layout* dst, int elem_bytes,
                 lm_plan** out) {
  return lm::plan_copy_impl(src, dst, elem_bytes, 0, 1, out);
}

int lm_plan_copy_shard(const lm_layout* src, const lm_layout* dst,
                       int elem_bytes, int rank, int world, lm_plan** out) {
  return lm::plan_copy_impl(src, dst, elem_bytes, rank, world, out);
}

int lm_plan_describe(const lm_plan* plan, char* buf, size_t cap) {
  if (!plan || (!buf && cap)) return LM_E_INVALID;
  if (cap == 0) return LM_E_BUFFER;
  const std::string& s = plan->describe;
  const size_t n = std::min(s.size(), cap - 1);
  std::memcpy(buf, s.data(), n);
  buf[n] = '\0';
  return s.size() + 1 > cap ? LM_E_BUFFER : LM_OK;
}

int lm_plan_extent(const lm_plan* plan, int64_t* size, int64_t* src_cosize,
                   int64_t* dst_cosize) {
  if (!plan) return LM_E_INVALID;
  if (size) *size = plan->size;
  if (src_cosize) *src_cosize = plan->src_cosize;
  if (dst_cosize) *dst_cosize = plan->dst_cosize;
  return LM_OK;
}

int lm_plan_launches(const lm_plan* plan, int* launches) {
  if (!plan || !launches) return LM_E_INVALID;
  *launches = int(plan->pieces.size());
  return LM_OK;
}

void lm_plan_destroy(lm_plan* plan) { delete plan; }

}  // extern "C"
