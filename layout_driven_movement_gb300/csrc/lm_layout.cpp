// Host layout algebra: construction, printing, evaluation, composition,
// zipped_divide, swizzle, concatenation, coalescing, right inverse and the
// common-vector search.  Pure C++17, no CUDA.
//
// Sources: "CUTE布局代数：GPU张量计算的内存优化革命" (§2.1 layouts, §2.2
// composition, §2.3 inverse and common sub-layout, §3.2 tiling, §4.2
// swizzle); "CUTLASS Layout可视化：从print_layout理解GPU内存映射与性能优化"
// (§2.1 offset formula, §3.2 notation, §3.3 coordinate order, §4.3 XOR
// swizzle); the PitchLinearStripminedThreadMap article (hotelren.com, §2.2).

#include <algorithm>
#include <cctype>
#include <cstring>
#include <limits>
#include <map>
#include <sstream>

#include "lm_internal.h"

namespace lm {

// ---------------------------------------------------------------------------
// flattening, size, cosize
// ---------------------------------------------------------------------------

static void flatten_into(const Node& n, std::vector<Leaf>& out) {
  if (n.leaf) {
    out.push_back({n.shape, n.stride});
    return;
  }
  for (const Node& k : n.kids) flatten_into(k, out);
}

std::vector<Leaf> flatten(const Node& n) {
  std::vector<Leaf> out;
  flatten_into(n, out);
  return out;
}

std::vector<Node> top_modes(const lm_layout& L) {
  if (L.root.leaf) return {L.root};
  return L.root.kids;
}

static void check_node(const Node& n, int depth) {
  if (depth > 64) fail(LM_E_INVALID);
  if (n.leaf) {
    if (n.shape < 0 || n.stride < 0) fail(LM_E_INVALID);
    return;
  }
  if (n.kids.empty()) fail(LM_E_INVALID);
  for (const Node& k : n.kids) check_node(k, depth + 1);
}

void finalize(lm_layout& L) {
  check_node(L.root, 0);
  L.leaves = flatten(L.root);
  L.mode_leaves.clear();
  for (const Node& m : top_modes(L))
    L.mode_leaves.push_back(int(flatten(m).size()));
  int64_t size = 1;
  bool empty = false;
  for (const Leaf& l : L.leaves) {
    if (l.e == 0) empty = true;
    else size = mul_chk(size, l.e);
  }
  if (empty) {
    L.size = 0;
    L.cosize = 0;
    return;
  }
  L.size = size;
  int64_t cos = 1;
  for (const Leaf& l : L.leaves) cos = add_chk(cos, mul_chk(l.e - 1, l.d));
  if (L.swz.on()) {
    const int64_t blk = int64_t(1) << (L.swz.m + L.swz.b);
    cos = mul_chk((cos + blk - 1) / blk, blk);
  }
  L.cosize = cos;
}

int64_t eval_affine(const std::vector<Leaf>& leaves, int64_t idx) {
  int64_t off = 0;
  for (const Leaf& l : leaves) {
    if (l.e == 1) continue;
    off += (idx % l.e) * l.d;
    idx /= l.e;
  }
  return off;
}

// ---------------------------------------------------------------------------
// printing and parsing ("CUTLASS Layout可视化" §3.2 notation)
// ---------------------------------------------------------------------------

static void print_node(const Node& n, bool shape, std::ostringstream& os) {
  if (n.leaf) {
    os << (shape ? n.shape : n.stride);
    return;
  }
  os << '(';
  for (size_t i = 0; i < n.kids.size(); ++i) {
    if (i) os << ',';
    print_node(n.kids[i], shape, os);
  }
  os << ')';
}

std::string to_string(const lm_layout& L) {
  std::ostringstream os;
  if (L.swz.on())
    os << "Sw<" << L.swz.b << ',' << L.swz.m << ',' << L.swz.s << "> o ";
  print_node(L.root, true, os);
  os << ':';
  print_node(L.root, false, os);
  return os.str();
}

namespace {
struct Parser {
  const char* p;
  void ws() {
    while (*p && std::isspace(static_cast<unsigned char>(*p))) ++p;
  }
  bool eat(char c) {
    ws();
    if (*p == c) {
      ++p;
      return true;
    }
    return false;
  }
  int64_t integer() {
    ws();
    if (*p == '_') ++p;
    if (!std::isdigit(static_cast<unsigned char>(*p))) fail(LM_E_INVALID);
    int64_t v = 0;
    while (std::isdigit(static_cast<unsigned char>(*p))) {
      v = add_chk(mul_chk(v, 10), *p - '0');
      ++p;
    }
    return v;
  }
  // tuple of integers; returns a Node whose leaves hold the integers in
  // .shape (the caller moves them into stride for the stride tuple)
  Node tuple() {
    ws();
    if (eat('(')) {
      std::vector<Node> kids;
      kids.push_back(tuple());
      while (eat(',')) kids.push_back(tuple());
      if (!eat(')')) fail(LM_E_INVALID);
      return Node::make_tuple(std::move(kids));
    }
    return Node::make_leaf(integer(), 0);
  }
};

bool same_structure(const Node& a, const Node& b) {
  if (a.leaf != b.leaf) return false;
  if (a.leaf) return true;
  if (a.kids.size() != b.kids.size()) return false;
  for (size_t i = 0; i < a.kids.size(); ++i)
    if (!same_structure(a.kids[i], b.kids[i])) return false;
  return true;
}

void merge_strides(Node& shape, const Node& stride) {
  if (shape.leaf) {
    shape.stride = stride.shape;
    return;
  }
  for (size_t i = 0; i < shape.kids.size(); ++i)
    merge_strides(shape.kids[i], stride.kids[i]);
}
}  // namespace

static lm_layout parse_layout(const char* text) {
  Parser ps{text};
  lm_layout L;
  ps.ws();
  if (std::strncmp(ps.p, "Sw<", 3) == 0) {
    ps.p += 3;
    L.swz.b = int32_t(ps.integer());
    if (!ps.eat(',')) fail(LM_E_INVALID);
    L.swz.m = int32_t(ps.integer());
    if (!ps.eat(',')) fail(LM_E_INVALID);
    L.swz.s = int32_t(ps.integer());
    if (!ps.eat('>')) fail(LM_E_INVALID);
    if (!ps.eat('o')) fail(LM_E_INVALID);
    // optional "_0 o" offset term as CuTe prints it
    const char* save = ps.p;
    ps.ws();
    if (*ps.p == '_' || *ps.p == '0') {
      int64_t off = ps.integer();
      if (off != 0 || !ps.eat('o')) ps.p = save;
    }
    if (L.swz.s < L.swz.b || L.swz.b + L.swz.m + L.swz.s > 40)
      fail(LM_E_INVALID);
  }
  Node shape = ps.tuple();
  if (!ps.eat(':')) fail(LM_E_INVALID);
  Node stride = ps.tuple();
  ps.ws();
  if (*ps.p) fail(LM_E_INVALID);
  if (!same_structure(shape, stride)) fail(LM_E_INVALID);
  merge_strides(shape, stride);
  L.root = std::move(shape);
  if (L.swz.b == 0) L.swz = Swz{};
  finalize(L);
  return L;
}

// ---------------------------------------------------------------------------
// coalescing and injectivity
// ---------------------------------------------------------------------------

std::vector<Leaf> coalesce_leaves(const std::vector<Leaf>& leaves) {
  std::vector<Leaf> out;
  for (const Leaf& l : leaves) {
    if (l.e == 0) return {{0, 0}};
    if (l.e == 1) continue;
    if (!out.empty() && l.d == out.back().e * out.back().d) {
      out.back().e = mul_chk(out.back().e, l.e);
      continue;
    }
    out.push_back(l);
  }
  return out;
}

// Sufficient test first: sorted by stride, every stride exceeds the largest
// offset the smaller-stride leaves reach (a mixed-radix number system).  If
// that fails, an exact bitmap check for small layouts; otherwise "not shown".
bool affine_injective(std::vector<Leaf> leaves) {
  std::vector<Leaf> ls;
  for (const Leaf& l : leaves) {
    if (l.e == 0) return true;
    if (l.e > 1) ls.push_back(l);
  }
  for (const Leaf& l : ls)
    if (l.d == 0) return false;
  std::sort(ls.begin(), ls.end(),
            [](const Leaf& a, const Leaf& b) { return a.d < b.d; });
  int64_t reach = 0;  // largest offset of the leaves so far
  bool radix = true;
  for (const Leaf& l : ls) {
    if (l.d <= reach) {
      radix = false;
      break;
    }
    reach = add_chk(reach, mul_chk(l.e - 1, l.d));
  }
  if (radix) return true;
  int64_t size = 1, cos = 1;
  for (const Leaf& l : ls) {
    size = mul_chk(size, l.e);
    cos = add_chk(cos, mul_chk(l.e - 1, l.d));
  }
  if (size > (int64_t(1) << 24) || cos > (int64_t(1) << 30)) return false;
  std::vector<uint64_t> bits(size_t((cos + 63) / 64), 0);
  for (int64_t i = 0; i < size; ++i) {
    int64_t o = eval_affine(ls, i);
    uint64_t& w = bits[size_t(o >> 6)];
    const uint64_t b = uint64_t(1) << (o & 63);
    if (w & b) return false;
    w |= b;
  }
  return true;
}

// ---------------------------------------------------------------------------
// composition ("CUTE布局代数" §2.2)
// ---------------------------------------------------------------------------

// A's leaves prepared for composition: coalesced, except that the literal
// last leaf keeps its own stride because past A's domain the last leaf keeps
// counting with that stride.
static std::vector<Leaf> outer_leaves(const std::vector<Leaf>& raw) {
  std::vector<Leaf> out;
  for (size_t i = 0; i < raw.size(); ++i) {
    const Leaf& l = raw[i];
    const bool last = (i + 1 == raw.size());
    if (l.e == 1 && !last) continue;
    // merging a leaf that continues the previous one keeps the function,
    // also for the extended last leaf: (q%e0)*d0 + (q/e0)*e0*d0 == q*d0
    if (!out.empty() && l.d == mul_chk(out.back().e, out.back().d)) {
      out.back().e = mul_chk(out.back().e, l.e);
      continue;
    }
    out.push_back(l);
  }
  if (out.empty()) out.push_back({1, 0});
  return out;
}

// A o (s:d) for one leaf of B: the leaves of the sub-layout it becomes.
// The last entry of `a` is unbounded (extends past its extent).
//
// A reads its argument as mixed-radix digits (one per leaf).  The values
// c*d, c < s, occupy a run of those digits, possibly starting inside a digit
// (a digit split by d) and ending inside one (a partial take).  `used[j]`
// accumulates, over all leaves of B, the largest value the leaves place in
// digit j; composing leaf by leaf is exact only while no digit overflows,
// i.e. while adding the leaves' values never carries (checked by the
// caller).
static std::vector<Leaf> compose_leaf(const std::vector<Leaf>& a_in,
                                      int64_t s, int64_t d,
                                      std::vector<int64_t>& used) {
  if (s == 0) return {{0, 0}};
  if (s == 1) return {{1, 0}};
  if (d == 0) return {{s, 0}};
  std::vector<Leaf> a = a_in;
  const size_t n = a.size();
  std::vector<int64_t> step(n, 1);  // digit value of one step of leaf a[j]
  size_t k = 0;
  int64_t rest = d;
  // divide out the stride d: skip whole digits, or split one
  while (k + 1 < n && rest > 1) {
    const int64_t e = a[k].e;
    if (rest % e == 0) {
      rest /= e;
      ++k;
    } else if (e % rest == 0) {
      a[k].e = e / rest;
      a[k].d = mul_chk(a[k].d, rest);
      step[k] = rest;
      rest = 1;
    } else {
      fail(LM_E_NOT_REPRESENTABLE);
    }
  }
  if (rest > 1) {  // k is the last digit: unbounded, just scale its stride
    a[k].d = mul_chk(a[k].d, rest);
    a[k].e = std::numeric_limits<int64_t>::max();
    step[k] = rest;
  }
  // take s consecutive coordinates
  std::vector<Leaf> out;
  int64_t rem = s;
  for (size_t j = k; j < n && rem > 1; ++j) {
    const bool last = (j + 1 == n);
    const int64_t e = last ? std::numeric_limits<int64_t>::max() : a[j].e;
    const int64_t take = rem <= e ? rem : e;
    if (rem > e && rem % e != 0) fail(LM_E_NOT_REPRESENTABLE);
    out.push_back({take, a[j].d});
    if (!last) used[j] = add_chk(used[j], mul_chk(take - 1, step[j]));
    rem = rem <= e ? 1 : rem / e;
  }
  std::vector<Leaf> co = coalesce_leaves(out);
  if (co.empty()) co.push_back({1, 0});
  return co;
}

static Node leaves_node(const std::vector<Leaf>& ls) {
  if (ls.size() == 1) return Node::make_leaf(ls[0].e, ls[0].d);
  std::vector<Node> kids;
  for (const Leaf& l : ls) kids.push_back(Node::make_leaf(l.e, l.d));
  return Node::make_tuple(std::move(kids));
}

static Node compose_node(const std::vector<Leaf>& a, const Node& b,
                         std::vector<int64_t>& used) {
  if (b.leaf) return leaves_node(compose_leaf(a, b.shape, b.stride, used));
  std::vector<Node> kids;
  for (const Node& k : b.kids) kids.push_back(compose_node(a, k, used));
  return Node::make_tuple(std::move(kids));
}

// no digit of A may receive more than it holds: then A(B(i)) is the sum of
// the per-leaf compositions
static void check_no_carry(const std::vector<Leaf>& a,
                           const std::vector<int64_t>& used) {
  for (size_t j = 0; j + 1 < a.size(); ++j)
    if (used[j] > a[j].e - 1) fail(LM_E_NOT_REPRESENTABLE);
}

static lm_layout compose(const lm_layout& A, const lm_layout& B) {
  if (B.swz.on() || A.size == 0) fail(LM_E_NOT_REPRESENTABLE);
  lm_layout R;
  const std::vector<Leaf> a = outer_leaves(A.leaves);
  std::vector<int64_t> used(a.size(), 0);
  R.root = compose_node(a, B.root, used);
  check_no_carry(a, used);
  R.swz = A.swz;
  finalize(R);
  return R;
}

// ---------------------------------------------------------------------------
// zipped_divide ("CUTE布局代数" §3.2)
// ---------------------------------------------------------------------------

static lm_layout zipped_divide(const lm_layout& L, int n,
                               const int64_t* tiler) {
  std::vector<Node> modes = top_modes(L);
  if (n != int(modes.size())) fail(LM_E_INVALID);
  std::vector<Node> tiles, rests;
  for (int k = 0; k < n; ++k) {
    const int64_t t = tiler[k];
    if (t < 1) fail(LM_E_INVALID);
    std::vector<Leaf> ml = flatten(modes[size_t(k)]);
    int64_t msize = 1;
    for (const Leaf& l : ml) msize = mul_chk(msize, l.e);
    if (msize % t != 0) fail(LM_E_NOT_REPRESENTABLE);
    // inside the mode's domain, so the mode's own (coalesced) leaves serve
    std::vector<Leaf> mc = coalesce_leaves(ml);
    if (mc.empty()) mc.push_back({1, 0});
    std::vector<int64_t> used(mc.size(), 0);
    tiles.push_back(leaves_node(compose_leaf(mc, t, 1, used)));
    rests.push_back(leaves_node(compose_leaf(mc, msize / t, t, used)));
    check_no_carry(mc, used);
  }
  lm_layout R;
  R.root = Node::make_tuple(
      {Node::make_tuple(std::move(tiles)), Node::make_tuple(std::move(rests))});
  R.swz = L.swz;
  finalize(R);
  if (R.size != L.size) fail(LM_E_NOT_REPRESENTABLE);
  return R;
}

// ---------------------------------------------------------------------------
// right inverse and common vector ("CUTE布局代数" §2.3)
// ---------------------------------------------------------------------------

static lm_layout right_inverse(const lm_layout& L) {
  if (L.swz.on()) fail(LM_E_NOT_REPRESENTABLE);
  struct Item {
    int64_t e, d, w;  // extent, stride, colex weight in L's domain
  };
  std::vector<Item> items;
  int64_t w = 1;
  for (const Leaf& l : L.leaves) {
    if (l.e > 1) items.push_back({l.e, l.d, w});
    w = mul_chk(w, std::max<int64_t>(l.e, 1));
  }
  std::stable_sort(items.begin(), items.end(),
                   [](const Item& a, const Item& b) { return a.d < b.d; });
  std::vector<Node> kids;
  int64_t expect = 1;
  for (size_t i = 0; i < items.size(); ++i) {
    const Item& it = items[i];
    if (it.d != expect) break;
    // a second leaf with the same stride makes the offsets ambiguous
    if (i + 1 < items.size() && items[i + 1].d == it.d) break;
    kids.push_back(Node::make_leaf(it.e, it.w));
    expect = mul_chk(expect, it.e);
  }
  lm_layout R;
  if (L.size == 0) {
    R.root = Node::make_leaf(0, 0);
  } else if (kids.empty()) {
    R.root = Node::make_leaf(1, 0);
  } else if (kids.size() == 1) {
    R.root = kids[0];
  } else {
    R.root = Node::make_tuple(std::move(kids));
  }
  finalize(R);
  return R;
}

// Exact brute force over inverse tables (small layouts).
static int64_t common_vector_brute(const lm_layout& A, const lm_layout& B) {
  const int64_t n = std::max(A.cosize, B.cosize);
  auto inv = [n](const lm_layout& L) {
    std::vector<int64_t> t(size_t(n), -1);
    for (int64_t i = 0; i < L.size; ++i) {
      int64_t o = L.swz.apply(eval_affine(L.leaves, i));
      int64_t& slot = t[size_t(o)];
      slot = (slot == -1) ? i : -2;
    }
    return t;
  };
  std::vector<int64_t> ia = inv(A), ib = inv(B);
  int64_t k = 0;
  while (k < n && ia[size_t(k)] >= 0 && ia[size_t(k)] == ib[size_t(k)]) ++k;
  return k;
}

// Common refinement of two leaf lists over the same colex domain: joint
// modes (e, s, d).  Returns false when the extents do not nest.
bool refine(const std::vector<Leaf>& sa, const std::vector<Leaf>& sb,
            std::vector<JMode>& out) {
  out.clear();
  std::vector<Leaf> a, b;
  for (const Leaf& l : sa)
    if (l.e != 1) a.push_back(l);
  for (const Leaf& l : sb)
    if (l.e != 1) b.push_back(l);
  size_t i = 0, j = 0;
  Leaf ca{1, 0}, cb{1, 0};
  if (i < a.size()) ca = a[i];
  if (j < b.size()) cb = b[j];
  while (i < a.size() && j < b.size()) {
    if (ca.e == cb.e) {
      out.push_back({ca.e, ca.d, cb.d});
      ++i;
      ++j;
      if (i < a.size()) ca = a[i];
      if (j < b.size()) cb = b[j];
    } else if (ca.e < cb.e) {
      if (cb.e % ca.e) return false;
      out.push_back({ca.e, ca.d, cb.d});
      cb.e /= ca.e;
      cb.d = mul_chk(cb.d, ca.e);
      ++i;
      if (i < a.size()) ca = a[i];
    } else {
      if (ca.e % cb.e) return false;
      out.push_back({cb.e, ca.d, cb.d});
      ca.e /= cb.e;
      ca.d = mul_chk(ca.d, cb.e);
      ++j;
      if (j < b.size()) cb = b[j];
    }
  }
  return i == a.size() && j == b.size();
}

// Largest k with A‡(j) == B‡(j) for all j < k, from the joint modes of two
// unswizzled layouts (exact; see the header).
static int64_t common_vector_joint(const std::vector<JMode>& modes) {
  std::vector<JMode> ms;
  for (const JMode& m : modes)
    if (m.e > 1) {
      if (m.s == 0 || m.d == 0) return 0;  // offset 0 has several preimages
      ms.push_back(m);
    }
  std::vector<bool> used(ms.size(), false);
  int64_t P = 1;
  for (;;) {
    int cand = -1, n_d = 0, n_s = 0;
    for (size_t k = 0; k < ms.size(); ++k) {
      if (used[k]) continue;
      if (ms[k].d == P) {
        ++n_d;
        cand = int(k);
      }
      if (ms[k].s == P) ++n_s;
    }
    if (n_d != 1 || n_s != 1 || ms[size_t(cand)].s != P) return P;
    used[size_t(cand)] = true;
    const int64_t next = mul_chk(P, ms[size_t(cand)].e);
    int64_t bound = next;
    for (size_t k = 0; k < ms.size(); ++k)
      if (!used[k]) bound = std::min(bound, std::min(ms[k].s, ms[k].d));
    if (bound < next) return bound;
    P = next;
  }
}

static int64_t max_common_vector(const lm_layout& A, const lm_layout& B) {
  if (A.size != B.size) fail(LM_E_INCOMPATIBLE);
  if (A.size == 0) return 0;
  const int64_t lim = int64_t(1) << 20;
  if (A.size <= lim && A.cosize <= 4 * lim && B.cosize <= 4 * lim)
    return common_vector_brute(A, B);
  std::vector<JMode> jm;
  if (!A.swz.on() && !B.swz.on() && refine(A.leaves, B.leaves, jm))
    return common_vector_joint(jm);
  // General case: walk offsets while both sides' inverses agree.  The
  // inverse of a swizzled layout at j is the affine inverse at Swz(j); the
  // affine inverse is read off the stride-sorted contiguous chain of leaves.
  auto chain_inverse = [](const lm_layout& L, int64_t o, int64_t& idx) {
    // returns false if o lies beyond the contiguous chain of L
    struct It {
      int64_t e, d, w;
    };
    std::vector<It> its;
    int64_t w = 1;
    for (const Leaf& l : L.leaves) {
      if (l.e > 1) its.push_back({l.e, l.d, w});
      w *= std::max<int64_t>(l.e, 1);
    }
    std::sort(its.begin(), its.end(),
              [](const It& a, const It& b) { return a.d < b.d; });
    int64_t expect = 1, r = o;
    idx = 0;
    for (const It& it : its) {
      if (it.d != expect) break;
      idx += (r % it.e) * it.w;
      r /= it.e;
      expect *= it.e;
    }
    return r == 0;
  };
  int64_t k = 0;
  const int64_t limit = std::min(A.cosize, B.cosize);
  while (k < limit && k < (int64_t(1) << 31)) {
    int64_t ia, ib;
    if (!chain_inverse(A, A.swz.apply(k), ia)) break;
    if (!chain_inverse(B, B.swz.apply(k), ib)) break;
    if (ia != ib) break;
    ++k;
  }
  return k;
}

// ---------------------------------------------------------------------------
// complement and products ("CUTE布局代数" §4.1)
// ---------------------------------------------------------------------------

// complement(A, M): the stride-sorted layout R such that (A, R) is one-to-one
// and reaches every offset below M when A's strides nest: walking A's leaves
// by increasing stride, each gap between the offsets A already reaches
// (current) and the next leaf's stride becomes a leaf of R, and a last leaf
// runs R up to M.
static std::vector<Leaf> complement_leaves(const lm_layout& A, int64_t M) {
  if (A.swz.on()) fail(LM_E_NOT_REPRESENTABLE);
  std::vector<Leaf> ls;
  for (const Leaf& l : A.leaves) {
    if (l.e == 0) fail(LM_E_NOT_REPRESENTABLE);
    if (l.e > 1 && l.d > 0) ls.push_back(l);
  }
  std::sort(ls.begin(), ls.end(), [](const Leaf& x, const Leaf& y) {
    return x.d < y.d || (x.d == y.d && x.e < y.e);
  });
  std::vector<Leaf> out;
  int64_t cur = 1;
  for (const Leaf& l : ls) {
    if (l.d < cur || l.d % cur) fail(LM_E_NOT_REPRESENTABLE);
    if (l.d / cur > 1) out.push_back({l.d / cur, cur});
    cur = mul_chk(l.e, l.d);
  }
  const int64_t rest = (M + cur - 1) / cur;
  if (rest > 1) out.push_back({rest, cur});
  std::vector<Leaf> co = coalesce_leaves(out);
  if (co.empty()) co.push_back({1, 0});
  return co;
}

static lm_layout complement(const lm_layout& A, int64_t M) {
  lm_layout R;
  R.root = leaves_node(complement_leaves(A, M));
  finalize(R);
  return R;
}

// logical_product(A, B) = (A, complement(A, size(A) * cosize(B)) o B)
static lm_layout logical_product(const lm_layout& A, const lm_layout& B) {
  if (A.swz.on() || B.swz.on()) fail(LM_E_NOT_REPRESENTABLE);
  const lm_layout C = complement(A, mul_chk(A.size, B.cosize));
  const lm_layout P = compose(C, B);
  lm_layout R;
  R.root = Node::make_tuple({A.root, P.root});
  finalize(R);
  return R;
}

// blocked_product(A, B): the modes of logical_product zipped, mode k being
// (A's mode k, the product's mode k): tiles A laid out in the order of B.
static lm_layout blocked_product(const lm_layout& A, const lm_layout& B) {
  if (A.swz.on() || B.swz.on()) fail(LM_E_NOT_REPRESENTABLE);
  const std::vector<Node> am = top_modes(A), bm = top_modes(B);
  if (am.size() != bm.size()) fail(LM_E_INVALID);
  const lm_layout C = complement(A, mul_chk(A.size, B.cosize));
  const lm_layout P = compose(C, B);
  const std::vector<Node> pm = top_modes(P);
  std::vector<Node> kids;
  for (size_t k = 0; k < am.size(); ++k)
    kids.push_back(Node::make_tuple({am[k], pm[k]}));
  lm_layout R;
  R.root = Node::make_tuple(std::move(kids));
  finalize(R);
  return R;
}

// ---------------------------------------------------------------------------
// local_partition ("CUTLASS Layout可视化" §5.3)
// ---------------------------------------------------------------------------

// True when the layout maps its domain one-to-one onto [0, size): its
// leaves, sorted by stride, have strides 1, e0, e0*e1, ...
bool compact_bijection(const std::vector<Leaf>& leaves) {
  std::vector<Leaf> ls;
  for (const Leaf& l : leaves)
    if (l.e > 1) ls.push_back(l);
  std::sort(ls.begin(), ls.end(),
            [](const Leaf& a, const Leaf& b) { return a.d < b.d; });
  int64_t next = 1;
  for (const Leaf& l : ls) {
    if (l.d != next) return false;
    next = mul_chk(next, l.e);
  }
  return true;
}

// The per-mode coordinate (a colex index into each top mode) that the thread
// layout maps to thread number t.
std::vector<int64_t> thread_coordinate(const lm_layout& thr, int64_t t) {
  if (thr.swz.on() || !compact_bijection(thr.leaves)) fail(LM_E_INVALID);
  if (t < 0 || t >= thr.size) fail(LM_E_INVALID);
  std::vector<int64_t> c;
  for (const Node& m : top_modes(thr)) {
    int64_t ck = 0, w = 1;
    for (const Leaf& l : flatten(m)) {
      if (l.e > 1) ck += ((t / l.d) % l.e) * w;
      w *= l.e;
    }
    c.push_back(ck);
  }
  return c;
}

// Thread t's part: zipped_divide by the thread layout's mode sizes, the tile
// mode fixed at the thread's coordinate.  Returns the rest mode (the
// values, no swizzle) and the tile mode's offset at the coordinate in *base.
static lm_layout local_partition(const lm_layout& L, const lm_layout& thr,
                                 int64_t t, int64_t* base) {
  const std::vector<int64_t> c = thread_coordinate(thr, t);
  const std::vector<Node> lm_modes = top_modes(L);
  const std::vector<Node> tm = top_modes(thr);
  if (tm.size() > lm_modes.size()) fail(LM_E_INVALID);
  std::vector<int64_t> tiler, cc;
  for (size_t k = 0; k < lm_modes.size(); ++k) {
    int64_t tk = 1;
    if (k < tm.size())
      for (const Leaf& l : flatten(tm[k])) tk = mul_chk(tk, l.e);
    tiler.push_back(tk);
    cc.push_back(k < c.size() ? c[k] : 0);
  }
  lm_layout A = L;
  A.swz = Swz{};
  finalize(A);
  const lm_layout Z = zipped_divide(A, int(tiler.size()), tiler.data());
  lm_layout tile, part;
  tile.root = Z.root.kids[0];
  part.root = Z.root.kids[1];
  finalize(tile);
  finalize(part);
  int64_t idx = 0, w = 1;
  for (size_t k = 0; k < cc.size(); ++k) {
    idx += cc[k] * w;
    w *= tiler[k];
  }
  *base = eval_affine(tile.leaves, idx);
  return part;
}

static lm_layout stripmined(int64_t threads, int64_t pitch, int64_t strips,
                            int64_t k_row) {
  if (threads < 1 || pitch < 1 || strips < 1 || k_row < 1) fail(LM_E_INVALID);
  const int64_t group = mul_chk(pitch, strips);
  const int64_t groups = (threads + group - 1) / group;
  lm_layout L;
  L.root = Node::make_tuple(
      {Node::make_leaf(pitch, 1), Node::make_leaf(strips, k_row),
       Node::make_leaf(groups, mul_chk(group, k_row))});
  finalize(L);
  return L;
}

}  // namespace lm

// ===========================================================================
// C ABI
// ===========================================================================

using lm::Error;
using lm::fail;

namespace {
template <class F>
int guard(F&& f) {
  try {
    f();
    return LM_OK;
  } catch (const Error& e) {
    return e.status;
  } catch (const std::bad_alloc&) {
    return LM_E_NOMEM;
  } catch (...) {
    return LM_E_INVALID;
  }
}

lm_layout* publish(lm_layout&& L) { return new lm_layout(std::move(L)); }
}  // namespace

extern "C" {

int lm_layout_make(int n_leaves, const int64_t* shape, const int64_t* stride,
                   int n_modes, const int* leaves_per_mode, lm_layout** out) {
  if (out) *out = nullptr;
  return guard([&] {
    if (!out || n_leaves < 1 || n_leaves > 4096 || !shape || !stride ||
        n_modes < 0)
      fail(LM_E_INVALID);
    lm_layout L;
    if (n_modes == 0) {
      if (n_leaves != 1) fail(LM_E_INVALID);
      L.root = lm::Node::make_leaf(shape[0], stride[0]);
    } else {
      if (!leaves_per_mode) fail(LM_E_INVALID);
      std::vector<lm::Node> modes;
      int at = 0;
      for (int m = 0; m < n_modes; ++m) {
        const int c = leaves_per_mode[m];
        if (c < 1 || at + c > n_leaves) fail(LM_E_INVALID);
        if (c == 1) {
          modes.push_back(lm::Node::make_leaf(shape[at], stride[at]));
        } else {
          std::vector<lm::Node> kids;
          for (int i = 0; i < c; ++i)
            kids.push_back(lm::Node::make_leaf(shape[at + i], stride[at + i]));
          modes.push_back(lm::Node::make_tuple(std::move(kids)));
        }
        at += c;
      }
      if (at != n_leaves) fail(LM_E_INVALID);
      L.root = lm::Node::make_tuple(std::move(modes));
    }
    lm::finalize(L);
    *out = publish(std::move(L));
  });
}

int lm_layout_parse(const char* text, lm_layout** out) {
  if (out) *out = nullptr;
  return guard([&] {
    if (!text || !out) fail(LM_E_INVALID);
    *out = publish(lm::parse_layout(text));
  });
}

int lm_layout_to_string(const lm_layout* layout, char* buf, size_t cap) {
  return guard([&] {
    if (!layout || (!buf && cap)) fail(LM_E_INVALID);
    const std::string s = lm::to_string(*layout);
    if (cap == 0) fail(LM_E_BUFFER);
    const size_t n = std::min(s.size(), cap - 1);
    std::memcpy(buf, s.data(), n);
    buf[n] = '\0';
    if (s.size() + 1 > cap) fail(LM_E_BUFFER);
  });
}

int lm_layout_print_grid(const lm_layout* layout, int bank_elem_bytes,
                         char* buf, size_t cap) {
  return guard([&] {
    if (!layout || (!buf && cap)) fail(LM_E_INVALID);
    if (bank_elem_bytes < 0 || bank_elem_bytes > 16) fail(LM_E_INVALID);
    const std::vector<lm::Node> modes = lm::top_modes(*layout);
    if (modes.size() != 2) fail(LM_E_INVALID);
    const std::vector<lm::Leaf> l0 = lm::flatten(modes[0]),
                                l1 = lm::flatten(modes[1]);
    int64_t rows = 1, cols = 1;
    for (const lm::Leaf& l : l0) rows = lm::mul_chk(rows, l.e);
    for (const lm::Leaf& l : l1) cols = lm::mul_chk(cols, l.e);
    if (lm::mul_chk(rows, cols) > (int64_t(1) << 16)) fail(LM_E_INVALID);
    std::vector<int64_t> v(size_t(rows * cols));
    size_t width = 1;
    for (int64_t r = 0; r < rows; ++r)
      for (int64_t c = 0; c < cols; ++c) {
        int64_t o = layout->swz.apply(lm::eval_affine(l0, r) +
                                      lm::eval_affine(l1, c));
        if (bank_elem_bytes) o = (o * bank_elem_bytes / 4) % 32;
        v[size_t(r * cols + c)] = o;
        width = std::max(width, std::to_string(o).size());
      }
    std::string s;
    for (int64_t r = 0; r < rows; ++r) {
      for (int64_t c = 0; c < cols; ++c) {
        const std::string t = std::to_string(v[size_t(r * cols + c)]);
        if (c) s += ' ';
        s += std::string(width - t.size(), ' ') + t;
      }
      s += '\n';
    }
    if (cap == 0) fail(LM_E_BUFFER);
    const size_t n = std::min(s.size(), cap - 1);
    std::memcpy(buf, s.data(), n);
    buf[n] = '\0';
    if (s.size() + 1 > cap) fail(LM_E_BUFFER);
  });
}

int lm_layout_size(const lm_layout* layout, int64_t* size) {
  return guard([&] {
    if (!layout || !size) fail(LM_E_INVALID);
    *size = layout->size;
  });
}

int lm_layout_cosize(const lm_layout* layout, int64_t* cosize) {
  return guard([&] {
    if (!layout || !cosize) fail(LM_E_INVALID);
    *cosize = layout->cosize;
  });
}

int lm_layout_rank(const lm_layout* layout, int* n_modes, int* n_leaves) {
  return guard([&] {
    if (!layout) fail(LM_E_INVALID);
    if (n_modes) *n_modes = int(layout->mode_leaves.size());
    if (n_leaves) *n_leaves = int(layout->leaves.size());
  });
}

int lm_layout_leaves(const lm_layout* layout, int64_t* shape, int64_t* stride,
                     int* leaves_per_mode) {
  return guard([&] {
    if (!layout) fail(LM_E_INVALID);
    for (size_t i = 0; i < layout->leaves.size(); ++i) {
      if (shape) shape[i] = layout->leaves[i].e;
      if (stride) stride[i] = layout->leaves[i].d;
    }
    if (leaves_per_mode)
      for (size_t i = 0; i < layout->mode_leaves.size(); ++i)
        leaves_per_mode[i] = layout->mode_leaves[i];
  });
}

int lm_layout_get_swizzle(const lm_layout* layout, int* b, int* m, int* s) {
  return guard([&] {
    if (!layout) fail(LM_E_INVALID);
    if (b) *b = layout->swz.b;
    if (m) *m = layout->swz.m;
    if (s) *s = layout->swz.s;
  });
}

int lm_layout_eval(const lm_layout* layout, int64_t index, int64_t* offset) {
  return guard([&] {
    if (!layout || !offset || index < 0 || index >= layout->size)
      fail(LM_E_INVALID);
    *offset = layout->swz.apply(lm::eval_affine(layout->leaves, index));
  });
}

int lm_layout_eval_coord(const lm_layout* layout, int n,
                         const int64_t* leaf_coord, int64_t* offset) {
  return guard([&] {
    if (!layout || !offset || n != int(layout->leaves.size()) ||
        (n && !leaf_coord))
      fail(LM_E_INVALID);
    int64_t off = 0;
    for (int k = 0; k < n; ++k) {
      if (leaf_coord[k] < 0) fail(LM_E_INVALID);
      off = lm::add_chk(off, lm::mul_chk(leaf_coord[k], layout->leaves[size_t(k)].d));
    }
    *offset = layout->swz.apply(off);
  });
}

int lm_layout_compose(const lm_layout* a, const lm_layout* b, lm_layout** r) {
  if (r) *r = nullptr;
  return guard([&] {
    if (!a || !b || !r) fail(LM_E_INVALID);
    *r = publish(lm::compose(*a, *b));
  });
}

int lm_layout_zipped_divide(const lm_layout* layout, int n,
                            const int64_t* tiler, lm_layout** r) {
  if (r) *r = nullptr;
  return guard([&] {
    if (!layout || !r || n < 1 || !tiler) fail(LM_E_INVALID);
    *r = publish(lm::zipped_divide(*layout, n, tiler));
  });
}

int lm_layout_swizzle(const lm_layout* layout, int b, int m, int s,
                      lm_layout** r) {
  if (r) *r = nullptr;
  return guard([&] {
    if (!layout || !r || b < 0 || m < 0 || s < b || b + m + s > 40)
      fail(LM_E_INVALID);
    if (layout->swz.on()) fail(LM_E_NOT_REPRESENTABLE);
    lm_layout R = *layout;
    R.swz = (b == 0) ? lm::Swz{} : lm::Swz{b, m, s};
    lm::finalize(R);
    *r = publish(std::move(R));
  });
}

int lm_layout_concat(const lm_layout* a, const lm_layout* b, lm_layout** r) {
  if (r) *r = nullptr;
  return guard([&] {
    if (!a || !b || !r) fail(LM_E_INVALID);
    if (a->swz.on() || b->swz.on()) fail(LM_E_NOT_REPRESENTABLE);
    lm_layout R;
    R.root = lm::Node::make_tuple({a->root, b->root});
    lm::finalize(R);
    *r = publish(std::move(R));
  });
}

int lm_layout_coalesce(const lm_layout* layout, lm_layout** r) {
  if (r) *r = nullptr;
  return guard([&] {
    if (!layout || !r) fail(LM_E_INVALID);
    std::vector<lm::Leaf> c = lm::coalesce_leaves(layout->leaves);
    lm_layout R;
    if (c.empty()) c.push_back({1, 0});
    if (c.size() == 1) {
      R.root = lm::Node::make_leaf(c[0].e, c[0].d);
    } else {
      std::vector<lm::Node> kids;
      for (const lm::Leaf& l : c) kids.push_back(lm::Node::make_leaf(l.e, l.d));
      R.root = lm::Node::make_tuple(std::move(kids));
    }
    R.swz = layout->swz;
    lm::finalize(R);
    *r = publish(std::move(R));
  });
}

int lm_layout_right_inverse(const lm_layout* layout, lm_layout** r) {
  if (r) *r = nullptr;
  return guard([&] {
    if (!layout || !r) fail(LM_E_INVALID);
    *r = publish(lm::right_inverse(*layout));
  });
}

int lm_layout_max_common_vector(const lm_layout* a, const lm_layout* b,
                                int64_t* k) {
  return guard([&] {
    if (!a || !b || !k) fail(LM_E_INVALID);
    *k = lm::max_common_vector(*a, *b);
  });
}

int lm_layout_complement(const lm_layout* layout, int64_t cotarget,
                         lm_layout** r) {
  if (r) *r = nullptr;
  return guard([&] {
    if (!layout || !r || cotarget < 1) fail(LM_E_INVALID);
    *r = publish(lm::complement(*layout, cotarget));
  });
}

int lm_layout_logical_product(const lm_layout* a, const lm_layout* b,
                              lm_layout** r) {
  if (r) *r = nullptr;
  return guard([&] {
    if (!a || !b || !r) fail(LM_E_INVALID);
    *r = publish(lm::logical_product(*a, *b));
  });
}

int lm_layout_blocked_product(const lm_layout* a, const lm_layout* b,
                              lm_layout** r) {
  if (r) *r = nullptr;
  return guard([&] {
    if (!a || !b || !r) fail(LM_E_INVALID);
    *r = publish(lm::blocked_product(*a, *b));
  });
}

int lm_layout_local_partition(const lm_layout* layout, const lm_layout* thr,
                              int64_t thr_idx, lm_layout** part,
                              int64_t* base) {
  if (part) *part = nullptr;
  return guard([&] {
    if (!layout || !thr || !part || !base) fail(LM_E_INVALID);
    int64_t b = 0;
    lm_layout P = lm::local_partition(*layout, *thr, thr_idx, &b);
    *base = b;
    *part = publish(std::move(P));
  });
}

int lm_layout_stripmined(int64_t threads, int64_t pitch, int64_t strips,
                         int64_t k_row, lm_layout** r) {
  if (r) *r = nullptr;
  return guard([&] {
    if (!r) fail(LM_E_INVALID);
    *r = publish(lm::stripmined(threads, pitch, strips, k_row));
  });
}

void lm_layout_destroy(lm_layout* layout) { delete layout; }

const char* lm_status_string(int status) {
  switch (status) {
    case LM_OK: return "LM_OK";
    case LM_E_INVALID: return "LM_E_INVALID";
    case LM_E_INCOMPATIBLE: return "LM_E_INCOMPATIBLE";
    case LM_E_NOT_REPRESENTABLE: return "LM_E_NOT_REPRESENTABLE";
    case LM_E_NOT_INJECTIVE: return "LM_E_NOT_INJECTIVE";
    case LM_E_OVERFLOW: return "LM_E_OVERFLOW";
    case LM_E_CAPACITY: return "LM_E_CAPACITY";
    case LM_E_OVERLAP: return "LM_E_OVERLAP";
    case LM_E_CUDA: return "LM_E_CUDA";
    case LM_E_TIMEOUT: return "LM_E_TIMEOUT";
    case LM_E_NOMEM: return "LM_E_NOMEM";
    case LM_E_BUFFER: return "LM_E_BUFFER";
    default: return "LM_E_UNKNOWN";
  }
}

const char* lm_version(void) { return "0.1.0"; }

}  // extern "C"
