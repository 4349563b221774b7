// Host planning of the thread-value partitioned tile copy.
//
// The source and destination layouts share a domain (tile, grid...): mode 0
// is the tile (a tuple of tile modes, as zipped_divide produces), the other
// top modes number the tiles.  The shared layout covers one tile.  Each
// phase (source -> shared, shared -> destination) groups `vec` consecutive
// coordinates of one tile mode into a vector and gives thread t the
// local_partition of the grouped tile by the phase's thread layout
// ("CUTLASS Layout可视化" §5.3).  The plan stores, per phase, the thread
// layout's leaves with the offset step of each leaf coordinate and a table
// of value offsets, and checks exhaustively that every (thread, value)
// offset is base(t) + val(v) -- the affine split the device side relies on.

#include <algorithm>
#include <climits>
#include <cstring>
#include <sstream>
#include <string>
#include <vector>

#include "lm_internal.h"

namespace lm {

bool refine(const std::vector<Leaf>& a, const std::vector<Leaf>& b,
            std::vector<JMode>& out);  // lm_layout.cpp

namespace {

constexpr int64_t kMaxSmemBytes = 232448;  // opt-in shared memory per block
constexpr int64_t kMaxTileElems = 1 << 18;

// The tile modes of a layout over (tile, grid...): mode 0's own modes.
std::vector<Node> tile_modes(const lm_layout& L) {
  const std::vector<Node> top = top_modes(L);
  const Node& t = top[0];
  if (t.leaf) return {t};
  return t.kids;
}

int64_t node_size(const Node& n) {
  int64_t s = 1;
  for (const Leaf& l : flatten(n)) s = mul_chk(s, l.e);
  return s;
}

// Affine offsets (no swizzle) of every tile element, colex over the tile
// modes.
std::vector<int64_t> tile_offsets(const std::vector<Node>& modes) {
  std::vector<std::vector<Leaf>> ml;
  std::vector<int64_t> n;
  int64_t total = 1;
  for (const Node& m : modes) {
    ml.push_back(flatten(m));
    n.push_back(node_size(m));
    total = mul_chk(total, n.back());
  }
  if (total > kMaxTileElems) fail(LM_E_INVALID);
  std::vector<int64_t> out(static_cast<size_t>(total));
  for (int64_t i = 0; i < total; ++i) {
    int64_t rem = i, off = 0;
    for (size_t k = 0; k < modes.size(); ++k) {
      off = add_chk(off, eval_affine(ml[k], rem % n[k]));
      rem /= n[k];
    }
    out[size_t(i)] = off;
  }
  return out;
}

struct Side {
  std::vector<int64_t> off;  // tile element -> element offset
  Swz swz;
  std::vector<int64_t> grid_strides;  // global sides: strides of the grid
};

// Can `v` consecutive coordinates of tile mode g move as one vector on
// this side?  Runs must be unit-stride and start on a multiple of v, grid
// strides multiples of v, and the swizzle must keep 2^M-element runs.
bool vector_ok(const Side& s, const std::vector<int64_t>& n, int g,
               int64_t v) {
  if (v == 1) return true;
  if (n[size_t(g)] % v) return false;
  if (s.swz.on() && (int64_t(1) << s.swz.m) < v) return false;
  for (int64_t gs : s.grid_strides)
    if (gs % v) return false;
  int64_t before = 1;  // colex weight of mode g
  for (int k = 0; k < g; ++k) before *= n[size_t(k)];
  const int64_t total = int64_t(s.off.size());
  for (int64_t i = 0; i < total; ++i) {
    const int64_t xg = (i / before) % n[size_t(g)];
    if (xg % v) continue;
    const int64_t o = s.off[size_t(i)];
    if (o % v) return false;
    for (int64_t u = 1; u < v; ++u)
      if (s.off[size_t(i + u * before)] != o + u) return false;
  }
  return true;
}

// Fill one phase: `from` and `to` sides over the tile, thread layout thr.
// Returns LM_OK or the status of the first check that failed.
int plan_phase(const Side& from, const Side& to, const std::vector<int64_t>& n,
               const lm_layout& thr, int eb, int vec_bytes_req,
               lm_tv_phase& P, int* g_out, int want_g = -1) {
  if (thr.swz.on() || !compact_bijection(thr.leaves)) return LM_E_INVALID;
  if (thr.size < 1 || thr.size > 1024) return LM_E_INVALID;
  const std::vector<Node> tm = top_modes(thr);
  const int r = int(n.size());
  if (int(tm.size()) > r) return LM_E_INVALID;
  std::vector<int64_t> T(size_t(r), 1);
  for (size_t k = 0; k < tm.size(); ++k) T[k] = node_size(tm[k]);

  // candidate vectors: widest first
  std::vector<std::pair<int, int64_t>> cands;
  const int64_t vmax = std::max<int64_t>(1, 16 / eb);
  if (vec_bytes_req > 0) {
    if (vec_bytes_req % eb || vec_bytes_req / eb > vmax) return LM_E_INVALID;
    for (int g = 0; g < r; ++g) cands.push_back({g, vec_bytes_req / eb});
  } else {
    for (int64_t v = vmax; v >= 1; v /= 2)
      for (int g = 0; g < r; ++g) cands.push_back({g, v});
  }
  int g = -1;
  int64_t v = 1;
  for (auto [cg, cv] : cands) {
    if (want_g >= 0 && cg != want_g) continue;
    bool fits = true;
    for (int k = 0; k < r; ++k) {
      const int64_t units = k == cg ? n[size_t(k)] / cv : n[size_t(k)];
      if ((k == cg && n[size_t(k)] % cv) || units % T[size_t(k)]) fits = false;
    }
    if (!fits || !vector_ok(from, n, cg, cv) || !vector_ok(to, n, cg, cv))
      continue;
    g = cg;
    v = cv;
    break;
  }
  if (g < 0) return LM_E_NOT_REPRESENTABLE;

  std::vector<int64_t> units(n), rest(static_cast<size_t>(r));
  units[size_t(g)] /= v;
  int64_t n_val = 1;
  for (int k = 0; k < r; ++k) {
    rest[size_t(k)] = units[size_t(k)] / T[size_t(k)];
    n_val *= rest[size_t(k)];
  }
  if (n_val > LM_TV_MAX_VALUES) return LM_E_INVALID;
  const int64_t n_thr = thr.size;

  // element index of (thread coordinate c, value r) in the tile
  std::vector<std::vector<int64_t>> coords(static_cast<size_t>(n_thr));
  for (int64_t t = 0; t < n_thr; ++t) {
    coords[size_t(t)] = thread_coordinate(thr, t);
    coords[size_t(t)].resize(size_t(r), 0);
  }
  auto element = [&](int64_t t, int64_t val) {
    int64_t idx = 0, w = 1;
    for (int k = 0; k < r; ++k) {
      const int64_t rk = val % rest[size_t(k)];
      val /= rest[size_t(k)];
      int64_t x = coords[size_t(t)][size_t(k)] + T[size_t(k)] * rk;
      if (k == g) x *= v;
      idx += x * w;
      w *= n[size_t(k)];
    }
    return idx;
  };
  // base(t) and val(v) per side; check the split exhaustively
  std::vector<int64_t> bf(static_cast<size_t>(n_thr));
  std::vector<int64_t> bt(static_cast<size_t>(n_thr));
  for (int64_t t = 0; t < n_thr; ++t) {
    const int64_t e = element(t, 0);
    bf[size_t(t)] = from.off[size_t(e)];
    bt[size_t(t)] = to.off[size_t(e)];
  }
  std::vector<int64_t> vf(static_cast<size_t>(n_val));
  std::vector<int64_t> vt(static_cast<size_t>(n_val));
  for (int64_t q = 0; q < n_val; ++q) {
    const int64_t e = element(0, q);
    vf[size_t(q)] = from.off[size_t(e)] - bf[0];
    vt[size_t(q)] = to.off[size_t(e)] - bt[0];
  }
  for (int64_t t = 0; t < n_thr; ++t)
    for (int64_t q = 0; q < n_val; ++q) {
      const int64_t e = element(t, q);
      if (from.off[size_t(e)] != bf[size_t(t)] + vf[size_t(q)] ||
          to.off[size_t(e)] != bt[size_t(t)] + vt[size_t(q)])
        return LM_E_NOT_REPRESENTABLE;
    }
  // base(t) as a sum over the thread layout's leaves
  std::vector<Leaf> tl;
  for (const Leaf& l : thr.leaves)
    if (l.e > 1) tl.push_back(l);
  if (int(tl.size()) > LM_TV_MAX_THR_LEAVES) return LM_E_INVALID;
  std::vector<int64_t> sf(tl.size()), st(tl.size());
  for (size_t j = 0; j < tl.size(); ++j) {
    sf[j] = bf[size_t(tl[j].d)] - bf[0];
    st[j] = bt[size_t(tl[j].d)] - bt[0];
  }
  for (int64_t t = 0; t < n_thr; ++t) {
    int64_t f = bf[0], h = bt[0];
    for (size_t j = 0; j < tl.size(); ++j) {
      const int64_t c = (t / tl[j].d) % tl[j].e;
      f += c * sf[j];
      h += c * st[j];
    }
    if (f != bf[size_t(t)] || h != bt[size_t(t)]) return LM_E_NOT_REPRESENTABLE;
  }
  auto fits32 = [](int64_t x) { return x >= INT32_MIN && x <= INT32_MAX; };
  P = lm_tv_phase{};
  P.n_thr = int32_t(n_thr);
  P.n_val = int32_t(n_val);
  P.vec_bytes = int32_t(v * eb);
  P.n_leaves = int32_t(tl.size());
  // the device side works in bytes
  for (size_t j = 0; j < tl.size(); ++j) {
    const int64_t a = mul_chk(sf[j], eb), b = mul_chk(st[j], eb);
    if (!fits32(a) || !fits32(b)) return LM_E_OVERFLOW;
    P.leaf_ext[j] = int32_t(tl[j].e);
    P.leaf_stride[j] = int32_t(tl[j].d);
    P.from_step[j] = int32_t(a);
    P.to_step[j] = int32_t(b);
  }
  for (int64_t q = 0; q < n_val; ++q) {
    // base(0) is folded into the value table
    const int64_t a = mul_chk(vf[size_t(q)] + bf[0], eb);
    const int64_t b = mul_chk(vt[size_t(q)] + bt[0], eb);
    if (!fits32(a) || !fits32(b)) return LM_E_OVERFLOW;
    P.from_val[q] = int32_t(a);
    P.to_val[q] = int32_t(b);
  }
  *g_out = g;
  return LM_OK;
}

// A phase's thread layout when the caller gives none: the stripmined map of
// the PitchLinearStripminedThreadMap article (§2.2), Pitch and Strips chosen
// by the same search as lm_stripmined_tune (§4.1-§4.2: coalesced global
// segments first, then shared-memory wavefronts under the bank model).  The
// phase's global side fixes the row: its unit-stride tile mode a (mode 0 if
// none) holds the vectors of a row, the other mode b counts rows, ld apart
// in global memory.  A thread layout must tile a contiguous block
// (local_partition), which the stripmined map does when one Pitch x Strips
// group holds every thread, so only those candidates are searched: the
// thread layout is (P, S):(1, P) over (a, b), P threads along a row and S
// rows.  Up to 256 threads; fewer when the tile has fewer vectors or no
// candidate divides it.  Tiles of rank 1 or 2 only.
struct TunedThreads {
  lm_layout thr;
  int mode = 0;        // a, the vector mode
  int64_t vec = 1;     // elements per vector
  int64_t pitch = 0, strips = 0, segments = 0, wavefronts = 0;
};

TunedThreads default_threads(const Side& global, const Side& shared,
                             const std::vector<int64_t>& n,
                             const lm_layout& smem, int eb, int vec_bytes_req) {
  const int r = int(n.size());
  if (r < 1 || r > 2) fail(LM_E_INVALID);
  TunedThreads T;
  // the global side's unit-stride mode
  int a = 0;
  int64_t before = 1;
  for (int k = 0; k < r; ++k) {
    if (n[size_t(k)] > 1 &&
        global.off[size_t(before)] - global.off[0] == 1) {
      a = k;
      break;
    }
    before *= n[size_t(k)];
  }
  const int b = r == 2 ? 1 - a : -1;
  const int64_t k_row = n[size_t(a)];
  const int64_t rows = b >= 0 ? n[size_t(b)] : 1;
  int64_t ld = k_row;
  if (b >= 0) {
    const int64_t wb = b == 0 ? 1 : n[0];
    ld = std::max(k_row, global.off[size_t(wb)] - global.off[0]);
  }
  // the widest vector along a that both sides take
  const int64_t vmax = std::max<int64_t>(1, 16 / eb);
  int64_t v = 0;
  for (int64_t c = vmax; c >= 1; c /= 2) {
    if (vec_bytes_req > 0 && c * eb != vec_bytes_req) continue;
    if (k_row % c == 0 && vector_ok(global, n, a, c) &&
        vector_ok(shared, n, a, c)) {
      v = c;
      break;
    }
  }
  if (v == 0) fail(LM_E_NOT_REPRESENTABLE);
  // the shared layout seen as (rows, k_row)
  lm_layout view;
  const std::vector<Node> sm = top_modes(smem);
  if (r == 1)
    view.root = Node::make_tuple({Node::make_leaf(1, 0), sm[0]});
  else
    view.root = Node::make_tuple({sm[size_t(b)], sm[size_t(a)]});
  view.swz = smem.swz;
  finalize(view);
  int64_t units = (k_row / v) * rows, threads = 1;
  while (threads * 2 <= std::min<int64_t>(256, units)) threads *= 2;
  int rc = LM_E_NOT_REPRESENTABLE;
  for (; threads >= 1 && rc != LM_OK; threads /= 2)
    rc = stripmined_search(threads, k_row, rows, ld, eb, int(v), &view, true,
                           &T.pitch, &T.strips, &T.segments, &T.wavefronts);
  if (rc != LM_OK) fail(rc);
  // (P, S):(1, P) over (a, b), written in the tile's mode order
  if (r == 1)
    T.thr.root = Node::make_leaf(T.pitch, 1);
  else if (a == 0)
    T.thr.root = Node::make_tuple(
        {Node::make_leaf(T.pitch, 1), Node::make_leaf(T.strips, T.pitch)});
  else
    T.thr.root = Node::make_tuple(
        {Node::make_leaf(T.strips, T.pitch), Node::make_leaf(T.pitch, 1)});
  finalize(T.thr);
  T.mode = a;
  T.vec = v;
  return T;
}

// Simulated shared-memory wavefronts of one tile for one phase's shared
// side (`from` when reading the tile, `to` when writing it).
int64_t phase_wavefronts(const lm_tv_phase& P, const Swz& z,
                         bool shared_is_to, int64_t* ideal) {
  int64_t total = 0, id = 0;
  std::vector<int64_t> addr(32);
  bool valid[32];
  for (int w0 = 0; w0 < P.n_thr; w0 += 32) {
    for (int q = 0; q < P.n_val; ++q) {
      int cnt = 0;
      for (int l = 0; l < 32; ++l) {
        const int t = w0 + l;
        valid[l] = t < P.n_thr;
        addr[size_t(l)] = 0;
        if (!valid[l]) continue;
        ++cnt;
        int64_t f = 0, h = 0;
        for (int j = 0; j < P.n_leaves; ++j) {
          const int64_t c = (t / P.leaf_stride[j]) % P.leaf_ext[j];
          f += c * P.from_step[j];
          h += c * P.to_step[j];
        }
        const int64_t o = shared_is_to ? h + P.to_val[q] : f + P.from_val[q];
        addr[size_t(l)] = z.apply(o);  // bytes, byte swizzle
      }
      total += warp_wavefronts(addr.data(), valid, P.vec_bytes);
      const int per = P.vec_bytes <= 4 ? 32 : 128 / P.vec_bytes;
      for (int p0 = 0; p0 < cnt; p0 += per)
        id += std::max<int64_t>(
            1, (int64_t(std::min(per, cnt - p0)) * P.vec_bytes + 127) / 128);
    }
  }
  *ideal = id;
  return total;
}

// A swizzle of element offsets as the same swizzle of byte offsets: the
// XORed bits move up by log2(eb), the shift stays.
Swz bytes_swz(const Swz& z, int eb) {
  Swz r = z;
  if (!z.on()) return r;
  int k = 0;
  while ((1 << k) < eb) ++k;
  r.m = z.m + k;
  return r;
}

void set_swz(int32_t* out, const Swz& z) {
  out[0] = z.b;
  out[1] = z.m;
  out[2] = z.s;
}

lm_tv_plan plan_tv(const lm_layout& src, const lm_layout& smem,
                   const lm_layout& dst, const lm_layout* thr_load,
                   const lm_layout* thr_store, int eb, int vec_load,
                   int vec_store) {
  if (eb != 1 && eb != 2 && eb != 4 && eb != 8 && eb != 16)
    fail(LM_E_INVALID);
  if (src.size != dst.size) fail(LM_E_INCOMPATIBLE);
  const std::vector<Node> tsrc = tile_modes(src), tdst = tile_modes(dst);
  const std::vector<Node> tsm = top_modes(smem);
  if (tsrc.size() != tdst.size() || tsrc.size() != tsm.size())
    fail(LM_E_INCOMPATIBLE);
  std::vector<int64_t> n;
  for (size_t k = 0; k < tsrc.size(); ++k) {
    n.push_back(node_size(tsrc[k]));
    if (node_size(tdst[k]) != n.back() || node_size(tsm[k]) != n.back())
      fail(LM_E_INCOMPATIBLE);
  }
  if (smem.size < 1) fail(LM_E_INVALID);
  if (!affine_injective(smem.leaves)) fail(LM_E_NOT_INJECTIVE);
  if (!affine_injective(dst.leaves)) fail(LM_E_NOT_INJECTIVE);
  const int64_t smem_bytes = (mul_chk(smem.cosize, eb) + 15) / 16 * 16;
  if (smem_bytes > kMaxSmemBytes) fail(LM_E_INVALID);

  // grid: the top modes after the tile, refined jointly
  std::vector<Leaf> gs, gd;
  {
    const std::vector<Node> ts = top_modes(src), td = top_modes(dst);
    for (size_t k = 1; k < ts.size(); ++k)
      for (const Leaf& l : flatten(ts[k])) gs.push_back(l);
    for (size_t k = 1; k < td.size(); ++k)
      for (const Leaf& l : flatten(td[k])) gd.push_back(l);
  }
  std::vector<JMode> grid;
  if (src.size == 0) {
    gs.clear();  // no tiles: nothing to refine
    gd.clear();
  }
  if (!gs.empty() || !gd.empty()) {
    if (gs.empty()) gs.push_back({1, 0});
    if (gd.empty()) gd.push_back({1, 0});
    if (!refine(gs, gd, grid)) fail(LM_E_INCOMPATIBLE);
  }
  std::vector<JMode> g2;
  for (const JMode& m : grid)
    if (m.e != 1) g2.push_back(m);
  if (int(g2.size()) > LM_TV_MAX_GRID) fail(LM_E_INVALID);

  lm_tv_plan P;
  lm_tv_args& A = P.args;
  A.elem_bytes = eb;
  A.smem_bytes = int32_t(smem_bytes);
  A.n_grid = int32_t(g2.size());
  A.n_tiles = 1;
  bool small = true;
  for (size_t k = 0; k < g2.size(); ++k) {
    A.grid_ext[k] = g2[k].e;
    A.grid_src[k] = mul_chk(g2[k].s, eb);
    A.grid_dst[k] = mul_chk(g2[k].d, eb);
    A.n_tiles = mul_chk(A.n_tiles, g2[k].e);
    if (g2[k].e >= (int64_t(1) << 31)) small = false;
  }
  A.grid_fast = small && A.n_tiles < (int64_t(1) << 32) ? 1 : 0;
  if (A.grid_fast)
    for (size_t k = 0; k < g2.size(); ++k) {
      const FastDiv f = make_fastdiv(uint32_t(g2[k].e));
      A.grid_div[k] = lm_tv_fastdiv{f.d, f.m, f.s1, f.s2};
    }
  int64_t tile_size = 1;
  for (int64_t x : n) tile_size *= x;
  if (tile_size == 0) fail(LM_E_INVALID);  // a tile holds elements
  if (src.size == 0) A.n_tiles = 0;
  set_swz(A.src_swz, bytes_swz(src.swz, eb));
  set_swz(A.smem_swz, bytes_swz(smem.swz, eb));
  set_swz(A.dst_swz, bytes_swz(dst.swz, eb));
  // a swizzle reads bits [M+S, M+S+B) and writes [M, M+B): a tile base that
  // is a multiple of 2^(B+M+S) leaves both alone
  auto commutes = [&](const int32_t* z, bool dst_side) {
    if (z[0] == 0) return 1;
    const int64_t blk = int64_t(1) << (z[0] + z[1] + z[2]);
    for (int k = 0; k < A.n_grid; ++k)
      if ((dst_side ? A.grid_dst[k] : A.grid_src[k]) % blk) return 0;
    return 1;
  };
  A.src_swz_tile = commutes(A.src_swz, false);
  A.dst_swz_tile = commutes(A.dst_swz, true);
  auto fits31 = [&](const std::vector<int64_t>& off) {
    for (int64_t o : off)
      if (o < 0 || o * eb >= (int64_t(1) << 31)) return false;
    return true;
  };

  Side S, M, D;
  S.off = tile_offsets(tsrc);
  S.swz = src.swz;
  for (const JMode& m : g2) S.grid_strides.push_back(m.s);
  M.off = tile_offsets(tsm);
  M.swz = smem.swz;
  D.off = tile_offsets(tdst);
  D.swz = dst.swz;
  for (const JMode& m : g2) D.grid_strides.push_back(m.d);

  A.offsets32 = fits31(S.off) && fits31(D.off) ? 1 : 0;
  int gl = 0, gsd = 0;
  // phases without a thread layout from the caller get the tuned one
  TunedThreads tl, ts;
  if (!thr_load) tl = default_threads(S, M, n, smem, eb, vec_load);
  if (!thr_store) ts = default_threads(D, M, n, smem, eb, vec_store);
  int rc = thr_load ? plan_phase(S, M, n, *thr_load, eb, vec_load, A.load, &gl)
                    : plan_phase(S, M, n, tl.thr, eb, int(tl.vec * eb),
                                 A.load, &gl, tl.mode);
  if (rc != LM_OK) fail(rc);
  rc = thr_store ? plan_phase(M, D, n, *thr_store, eb, vec_store, A.store, &gsd)
                 : plan_phase(M, D, n, ts.thr, eb, int(ts.vec * eb), A.store,
                              &gsd, ts.mode);
  if (rc != LM_OK) fail(rc);
  A.block_threads =
      int32_t((std::max(A.load.n_thr, A.store.n_thr) + 31) / 32 * 32);

  P.src_cosize = src.cosize;
  P.dst_cosize = dst.cosize;
  int64_t wl_ideal = 0, ws_ideal = 0;
  const Swz zb = bytes_swz(smem.swz, eb);
  const int64_t wl = phase_wavefronts(A.load, zb, true, &wl_ideal);
  const int64_t ws = phase_wavefronts(A.store, zb, false, &ws_ideal);
  auto tuned = [](const lm_layout* given, const TunedThreads& t) {
    std::ostringstream o;
    o << ",\"thr\":\"" << to_string(given ? *given : t.thr) << "\"";
    if (given)
      o << ",\"tuned\":false";
    else
      o << ",\"tuned\":true,\"pitch\":" << t.pitch << ",\"strips\":"
        << t.strips << ",\"segments\":" << t.segments;
    return o.str();
  };
  std::ostringstream os;
  os << "{\"path\":\"TV\",\"n_tiles\":" << A.n_tiles
     << ",\"tile_elems\":" << tile_size << ",\"smem_bytes\":" << A.smem_bytes
     << ",\"block_threads\":" << A.block_threads << ",\"load\":{\"threads\":"
     << A.load.n_thr << ",\"values\":" << A.load.n_val
     << ",\"vec_bytes\":" << A.load.vec_bytes << ",\"vec_mode\":" << gl
     << ",\"smem_wavefronts\":" << wl << ",\"smem_wavefronts_ideal\":"
     << wl_ideal << tuned(thr_load, tl)
     << "},\"store\":{\"threads\":" << A.store.n_thr
     << ",\"values\":" << A.store.n_val << ",\"vec_bytes\":"
     << A.store.vec_bytes << ",\"vec_mode\":" << gsd
     << ",\"smem_wavefronts\":" << ws << ",\"smem_wavefronts_ideal\":"
     << ws_ideal << tuned(thr_store, ts) << "}}";
  P.describe = os.str();
  return P;
}

}  // namespace
}  // namespace lm

extern "C" {

int lm_tv_plan_create(const lm_layout* src, const lm_layout* smem,
                      const lm_layout* dst, const lm_layout* thr_load,
                      const lm_layout* thr_store, int elem_bytes,
                      int vec_load_bytes, int vec_store_bytes,
                      lm_tv_plan** out) {
  if (out) *out = nullptr;
  if (!src || !smem || !dst || !out) return LM_E_INVALID;
  try {
    *out = new lm_tv_plan(lm::plan_tv(*src, *smem, *dst, thr_load, thr_store,
                                      elem_bytes, vec_load_bytes,
                                      vec_store_bytes));
    return LM_OK;
  } catch (const lm::Error& e) {
    return e.status;
  } catch (const std::bad_alloc&) {
    return LM_E_NOMEM;
  }
}

int lm_tv_plan_describe(const lm_tv_plan* plan, char* buf, size_t cap) {
  if (!plan || (!buf && cap)) return LM_E_INVALID;
  if (cap == 0) return LM_E_BUFFER;
  const std::string& s = plan->describe;
  const size_t n = std::min(s.size(), cap - 1);
  std::memcpy(buf, s.data(), n);
  buf[n] = '\0';
  return s.size() + 1 > cap ? LM_E_BUFFER : LM_OK;
}

int lm_tv_plan_args(const lm_tv_plan* plan, void* args, size_t cap) {
  if (!plan || !args) return LM_E_INVALID;
  if (cap < sizeof(lm_tv_args)) return LM_E_BUFFER;
  std::memcpy(args, &plan->args, sizeof(lm_tv_args));
  return LM_OK;
}

void lm_tv_plan_destroy(lm_tv_plan* plan) { delete plan; }

}  // extern "C"
