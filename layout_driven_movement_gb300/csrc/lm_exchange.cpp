// A relayout whose source and destination are both sharded across ranks:
// rank r holds the source elements of one range of the joint mode that is
// slowest in source memory and must produce the destination elements of one
// range of the joint mode slowest in destination memory (a row-sharded
// transpose: rows in, the transposed rows out).  Each pair of ranks shares
// the box where the two ranges meet; the sender packs its part of every box
// into a contiguous buffer (a layout copy), one all-to-all exchange moves
// the buffers, and the receiver unpacks each into its destination shard
// (another layout copy).  This file plans the boxes and the copies; the
// exchange itself is the caller's collective.

#include <algorithm>
#include <cstring>
#include <memory>
#include <sstream>
#include <string>
#include <vector>

#include "lm_internal.h"

namespace {

struct PeerCopy {
  int64_t count = 0;        // elements in the box
  int64_t base = 0;         // elements into the local shard buffer
  lm_plan* plan = nullptr;  // box <-> compact buffer
  std::vector<lm::JMode> box;
};

}  // namespace

struct lm_exchange {
  int eb = 1, rank = 0, world = 1;
  int in_mode = -1, out_mode = -1;
  std::vector<lm::JMode> modes;
  int64_t src_local = 0, dst_local = 0;  // elements of the shard buffers
  int64_t src_origin = 0, dst_origin = 0;  // global offsets of their starts
  std::vector<PeerCopy> send, recv;
  // when both modes split evenly, every box has the same shape and the
  // packs (unpacks) of all peers form one layout copy each
  lm_plan* pack_all = nullptr;
  lm_plan* unpack_all = nullptr;
  std::string describe;
  ~lm_exchange() {
    for (PeerCopy& p : send) lm_plan_destroy(p.plan);
    for (PeerCopy& p : recv) lm_plan_destroy(p.plan);
    lm_plan_destroy(pack_all);
    lm_plan_destroy(unpack_all);
  }
};

namespace lm {
namespace {

// A layout of the given leaves, one top mode per leaf.
lm_layout leaves_layout(const std::vector<std::pair<int64_t, int64_t>>& ls) {
  lm_layout L;
  std::vector<Node> kids;
  for (const auto& l : ls) kids.push_back(Node::make_leaf(l.first, l.second));
  if (kids.empty()) kids.push_back(Node::make_leaf(1, 0));
  L.root = Node::make_tuple(std::move(kids));
  finalize(L);
  return L;
}

// Plan the copy between a box (strides `side`) and its compact colex image.
lm_plan* box_plan(const std::vector<JMode>& box, bool side_is_dst, int eb) {
  std::vector<std::pair<int64_t, int64_t>> strided, compact;
  int64_t w = 1;
  for (const JMode& m : box) {
    strided.push_back({m.e, side_is_dst ? m.d : m.s});
    compact.push_back({m.e, w});
    w = mul_chk(w, m.e);
  }
  const lm_layout S = leaves_layout(strided), C = leaves_layout(compact);
  lm_plan* p = nullptr;
  const int rc = side_is_dst ? lm_plan_copy(&C, &S, eb, &p)
                             : lm_plan_copy(&S, &C, eb, &p);
  if (rc != LM_OK) fail(rc);
  return p;
}

// The packs of all peers as one copy: the shard's box with the out mode
// cut into (box extent, peer), the packed buffer peer-major with each box
// compact.  The unpacks likewise, the in mode cut into (box extent, peer).
// Only when every box has the same shape (both modes split evenly) and the
// two modes differ.
void plan_all(lm_exchange& X) {
  const std::vector<JMode>& ms = X.modes;
  const int ki = X.in_mode, ko = X.out_mode, w = X.world;
  if (ki == ko || ms[size_t(ki)].e % w || ms[size_t(ko)].e % w) return;
  std::vector<int64_t> x;
  for (const JMode& m : ms) x.push_back(m.e);
  x[size_t(ki)] /= w;
  x[size_t(ko)] /= w;
  std::vector<std::pair<int64_t, int64_t>> shard_s, shard_d, packed;
  int64_t cw = 1;
  for (size_t j = 0; j < ms.size(); ++j) {
    shard_s.push_back({x[j], ms[j].s});
    shard_d.push_back({x[j], ms[j].d});
    packed.push_back({x[j], cw});
    cw = mul_chk(cw, x[j]);
  }
  // pack: peer q steps along the out mode in the source
  std::vector<std::pair<int64_t, int64_t>> ps = shard_s, pd = packed;
  ps.push_back({w, mul_chk(x[size_t(ko)], ms[size_t(ko)].s)});
  pd.push_back({w, cw});
  // unpack: peer p steps along the in mode in the destination
  std::vector<std::pair<int64_t, int64_t>> us = packed, ud = shard_d;
  us.push_back({w, cw});
  ud.push_back({w, mul_chk(x[size_t(ki)], ms[size_t(ki)].d)});
  const lm_layout PS = leaves_layout(ps), PD = leaves_layout(pd);
  const lm_layout US = leaves_layout(us), UD = leaves_layout(ud);
  lm_plan *a = nullptr, *b = nullptr;
  if (lm_plan_copy(&PS, &PD, X.eb, &a) != LM_OK) return;
  if (lm_plan_copy(&US, &UD, X.eb, &b) != LM_OK) {
    lm_plan_destroy(a);
    return;
  }
  X.pack_all = a;
  X.unpack_all = b;
}

// The joint mode with the largest stride on one side, or -1 when that mode
// has fewer than `world` coordinates: the shards are ranges of exactly that
// mode, so a shorter one cannot be split over every rank, and falling back
// to a faster mode would give shard ranges that overlap in memory.
int slowest_mode(const std::vector<JMode>& ms, int world, bool dst_side) {
  int k = -1;
  for (int j = 0; j < int(ms.size()); ++j) {
    const int64_t sj = dst_side ? ms[size_t(j)].d : ms[size_t(j)].s;
    const int64_t sk = k < 0 ? -1 : (dst_side ? ms[size_t(k)].d : ms[size_t(k)].s);
    if (k < 0 || sj > sk) k = j;
  }
  if (k >= 0 && ms[size_t(k)].e < world) return -1;
  return k;
}

// Offsets the box of `ms` restricted by `lo/hi` on one mode reaches on one
// side: [first, last + 1).
void side_span(const std::vector<JMode>& ms, int k, int64_t lo, int64_t hi,
               bool dst_side, int64_t* first, int64_t* end) {
  int64_t f = 0, l = 0;
  for (int j = 0; j < int(ms.size()); ++j) {
    const int64_t st = dst_side ? ms[size_t(j)].d : ms[size_t(j)].s;
    const int64_t a = j == k ? lo : 0;
    const int64_t b = j == k ? hi : ms[size_t(j)].e;
    f = add_chk(f, mul_chk(a, st));
    l = add_chk(l, mul_chk(b - 1, st));
  }
  *first = f;
  *end = l + 1;
}

lm_exchange* plan_exchange(const lm_layout& src, const lm_layout& dst, int eb,
                           int rank, int world) {
  if (eb != 1 && eb != 2 && eb != 4 && eb != 8 && eb != 16)
    fail(LM_E_INVALID);
  if (world < 1 || rank < 0 || rank >= world) fail(LM_E_INVALID);
  if (src.size != dst.size) fail(LM_E_INCOMPATIBLE);
  if (src.swz.on() || dst.swz.on()) fail(LM_E_NOT_REPRESENTABLE);
  if (src.size == 0) fail(LM_E_INVALID);
  if (!affine_injective(dst.leaves)) fail(LM_E_NOT_INJECTIVE);
  auto X = std::make_unique<lm_exchange>();
  X->eb = eb;
  X->rank = rank;
  X->world = world;
  if (!joint_modes(src, dst, X->modes)) fail(LM_E_INCOMPATIBLE);
  const std::vector<JMode>& ms = X->modes;
  if (ms.empty()) fail(LM_E_INVALID);
  X->in_mode = slowest_mode(ms, world, false);
  X->out_mode = slowest_mode(ms, world, true);
  if (X->in_mode < 0 || X->out_mode < 0) fail(LM_E_INVALID);
  const int ki = X->in_mode, ko = X->out_mode;
  const int64_t ei = ms[size_t(ki)].e, eo = ms[size_t(ko)].e;
  auto in_lo = [&](int r) { return ei * r / world; };
  auto out_lo = [&](int r) { return eo * r / world; };

  int64_t s_end = 0, d_end = 0;
  side_span(ms, ki, in_lo(rank), in_lo(rank + 1), false, &X->src_origin,
            &s_end);
  side_span(ms, ko, out_lo(rank), out_lo(rank + 1), true, &X->dst_origin,
            &d_end);
  X->src_local = s_end - X->src_origin;
  X->dst_local = d_end - X->dst_origin;

  // the box where input range of rank p meets output range of rank q
  auto box = [&](int p, int q, std::vector<JMode>& b, int64_t* origin_s,
                 int64_t* origin_d) {
    b = ms;
    std::vector<int64_t> o(ms.size(), 0);
    int64_t lo = in_lo(p), hi = in_lo(p + 1);
    o[size_t(ki)] = lo;
    b[size_t(ki)].e = hi - lo;
    int64_t clo = out_lo(q), chi = out_lo(q + 1);
    if (ko == ki) {
      clo = std::max(clo, lo);
      chi = std::min(chi, hi);
      b[size_t(ko)].e = std::max<int64_t>(0, chi - clo);
    } else {
      b[size_t(ko)].e = chi - clo;
    }
    o[size_t(ko)] = clo;
    int64_t os = 0, od = 0;
    for (size_t j = 0; j < ms.size(); ++j) {
      os = add_chk(os, mul_chk(o[j], ms[j].s));
      od = add_chk(od, mul_chk(o[j], ms[j].d));
    }
    *origin_s = os;
    *origin_d = od;
    int64_t n = 1;
    for (const JMode& m : b) n = mul_chk(n, m.e);
    return n;
  };
  std::ostringstream os;
  os << "{\"rank\":" << rank << ",\"world\":" << world << ",\"modes\":[";
  for (size_t j = 0; j < ms.size(); ++j)
    os << (j ? "," : "") << '[' << ms[j].e << ',' << ms[j].s << ','
       << ms[j].d << ']';
  os << "],\"in_mode\":" << ki << ",\"out_mode\":" << ko
     << ",\"src_origin\":" << X->src_origin << ",\"src_local\":"
     << X->src_local << ",\"dst_origin\":" << X->dst_origin
     << ",\"dst_local\":" << X->dst_local;
  for (int dir = 0; dir < 2; ++dir) {
    os << (dir == 0 ? ",\"send\":[" : ",\"recv\":[");
    for (int peer = 0; peer < world; ++peer) {
      PeerCopy pc;
      int64_t org_s = 0, org_d = 0;
      const int p = dir == 0 ? rank : peer, q = dir == 0 ? peer : rank;
      pc.count = box(p, q, pc.box, &org_s, &org_d);
      if (pc.count > 0) {
        if (dir == 0) {
          pc.base = org_s - X->src_origin;
          pc.plan = box_plan(pc.box, false, eb);
        } else {
          pc.base = org_d - X->dst_origin;
          pc.plan = box_plan(pc.box, true, eb);
        }
      }
      os << (peer ? "," : "") << "{\"count\":" << pc.count
         << ",\"base\":" << pc.base << ",\"box\":[";
      for (size_t j = 0; j < pc.box.size(); ++j)
        os << (j ? "," : "") << '[' << pc.box[j].e << ',' << pc.box[j].s
           << ',' << pc.box[j].d << ']';
      os << "]}";
      (dir == 0 ? X->send : X->recv).push_back(std::move(pc));
    }
    os << ']';
  }
  plan_all(*X);
  os << ",\"one_copy_per_side\":" << (X->pack_all ? "true" : "false");
  os << '}';
  X->describe = os.str();
  return X.release();
}

}  // namespace
}  // namespace lm

extern "C" {

int lm_plan_exchange(const lm_layout* src, const lm_layout* dst,
                     int elem_bytes, int rank, int world, lm_exchange** out) {
  if (out) *out = nullptr;
  if (!src || !dst || !out) return LM_E_INVALID;
  try {
    *out = lm::plan_exchange(*src, *dst, elem_bytes, rank, world);
    return LM_OK;
  } catch (const lm::Error& e) {
    return e.status;
  } catch (const std::bad_alloc&) {
    return LM_E_NOMEM;
  }
}

int lm_exchange_describe(const lm_exchange* x, char* buf, size_t cap) {
  if (!x || (!buf && cap)) return LM_E_INVALID;
  if (cap == 0) return LM_E_BUFFER;
  const size_t n = std::min(x->describe.size(), cap - 1);
  std::memcpy(buf, x->describe.data(), n);
  buf[n] = '\0';
  return x->describe.size() + 1 > cap ? LM_E_BUFFER : LM_OK;
}

int lm_exchange_sizes(const lm_exchange* x, int64_t* src_local,
                      int64_t* dst_local, int64_t* send_counts,
                      int64_t* recv_counts) {
  if (!x) return LM_E_INVALID;
  if (src_local) *src_local = x->src_local;
  if (dst_local) *dst_local = x->dst_local;
  for (int p = 0; p < x->world; ++p) {
    if (send_counts) send_counts[p] = x->send[size_t(p)].count;
    if (recv_counts) recv_counts[p] = x->recv[size_t(p)].count;
  }
  return LM_OK;
}

int lm_exchange_pack(const lm_exchange* x, int peer, const void* src_local,
                     int64_t src_capacity_elems, void* send,
                     int64_t send_capacity_elems, void* cuda_stream) {
  if (!x || peer < 0 || peer >= x->world) return LM_E_INVALID;
  const PeerCopy& pc = x->send[size_t(peer)];
  if (pc.count == 0) return LM_OK;
  if (!src_local || !send) return LM_E_INVALID;
  if (src_capacity_elems < x->src_local) return LM_E_CAPACITY;
  const char* s = static_cast<const char*>(src_local) + pc.base * x->eb;
  return lm_layout_copy(pc.plan, s, src_capacity_elems - pc.base, send,
                        send_capacity_elems, cuda_stream);
}

int lm_exchange_unpack(const lm_exchange* x, int peer, const void* recv,
                       int64_t recv_capacity_elems, void* dst_local,
                       int64_t dst_capacity_elems, void* cuda_stream) {
  if (!x || peer < 0 || peer >= x->world) return LM_E_INVALID;
  const PeerCopy& pc = x->recv[size_t(peer)];
  if (pc.count == 0) return LM_OK;
  if (!recv || !dst_local) return LM_E_INVALID;
  if (dst_capacity_elems < x->dst_local) return LM_E_CAPACITY;
  char* d = static_cast<char*>(dst_local) + pc.base * x->eb;
  return lm_layout_copy(pc.plan, recv, recv_capacity_elems, d,
                        dst_capacity_elems - pc.base, cuda_stream);
}

int lm_exchange_pack_all(const lm_exchange* x, const void* src_local,
                         int64_t src_capacity_elems, void* send,
                         int64_t send_capacity_elems, void* cuda_stream) {
  if (!x) return LM_E_INVALID;
  if (!x->pack_all) {
    int64_t off = 0;
    for (int q = 0; q < x->world; ++q) {
      const int64_t n = x->send[size_t(q)].count;
      if (n && off + n > send_capacity_elems) return LM_E_CAPACITY;
      const int rc = lm_exchange_pack(
          x, q, src_local, src_capacity_elems,
          n ? static_cast<char*>(send) + off * x->eb : send, n, cuda_stream);
      if (rc != LM_OK) return rc;
      off += n;
    }
    return LM_OK;
  }
  if (src_capacity_elems < x->src_local) return LM_E_CAPACITY;
  return lm_layout_copy(x->pack_all, src_local, src_capacity_elems, send,
                        send_capacity_elems, cuda_stream);
}

int lm_exchange_unpack_all(const lm_exchange* x, const void* recv,
                           int64_t recv_capacity_elems, void* dst_local,
                           int64_t dst_capacity_elems, void* cuda_stream) {
  if (!x) return LM_E_INVALID;
  if (!x->unpack_all) {
    int64_t off = 0;
    for (int p = 0; p < x->world; ++p) {
      const int64_t n = x->recv[size_t(p)].count;
      if (n && off + n > recv_capacity_elems) return LM_E_CAPACITY;
      const int rc = lm_exchange_unpack(
          x, p, n ? static_cast<const char*>(recv) + off * x->eb : recv, n,
          dst_local, dst_capacity_elems, cuda_stream);
      if (rc != LM_OK) return rc;
      off += n;
    }
    return LM_OK;
  }
  if (dst_capacity_elems < x->dst_local) return LM_E_CAPACITY;
  return lm_layout_copy(x->unpack_all, recv, recv_capacity_elems, dst_local,
                        dst_capacity_elems, cuda_stream);
}

void lm_exchange_destroy(lm_exchange* x) { delete x; }

}  // extern "C"
