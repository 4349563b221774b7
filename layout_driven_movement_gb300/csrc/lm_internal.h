// Internal data structures of the layoutmove library: the layout tree, the
// lowered copy plan, and the plain-old-data argument blocks handed to the
// CUDA kernels.  Included by the host C++ files and by the .cu file.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "layoutmove.h"
#include "layoutmove_tv.h"

#if defined(__CUDACC__)
#define LM_HD __host__ __device__ __forceinline__
#else
#define LM_HD inline
#endif

namespace lm {

// ---------------------------------------------------------------------------
// Status handling: every internal failure throws Error(status); the C ABI
// catches it and returns the code.
// ---------------------------------------------------------------------------
struct Error {
  int status;
  explicit Error(int s) : status(s) {}
};

[[noreturn]] inline void fail(int status) { throw Error(status); }

inline int64_t mul_chk(int64_t a, int64_t b) {
  int64_t r;
  if (__builtin_mul_overflow(a, b, &r)) fail(LM_E_OVERFLOW);
  return r;
}
inline int64_t add_chk(int64_t a, int64_t b) {
  int64_t r;
  if (__builtin_add_overflow(a, b, &r)) fail(LM_E_OVERFLOW);
  return r;
}

// ---------------------------------------------------------------------------
// Swizzle<B,M,S>: o ^ ((o >> S) & ((2^B - 1) << M)).
// ---------------------------------------------------------------------------
struct Swz {
  int32_t b = 0, m = 0, s = 0;
  LM_HD bool on() const { return b > 0; }
  LM_HD int64_t apply(int64_t o) const {
    return b > 0 ? (o ^ ((o >> s) & (((int64_t(1) << b) - 1) << m))) : o;
  }
};

// ---------------------------------------------------------------------------
// Layout tree.  A node is a leaf (extent:stride) or a tuple of nodes.
// ---------------------------------------------------------------------------
struct Node {
  bool leaf = true;
  int64_t shape = 1;
  int64_t stride = 0;
  std::vector<Node> kids;

  static Node make_leaf(int64_t e, int64_t d) {
    Node n;
    n.leaf = true;
    n.shape = e;
    n.stride = d;
    return n;
  }
  static Node make_tuple(std::vector<Node> k) {
    Node n;
    n.leaf = false;
    n.kids = std::move(k);
    return n;
  }
};

struct Leaf {
  int64_t e;  // extent
  int64_t d;  // stride (elements)
};

}  // namespace lm

// The opaque handle of the C ABI.
struct lm_layout {
  lm::Node root;   // a leaf (integer layout) or a tuple of top-level modes
  lm::Swz swz;     // swizzle on the whole offset (b == 0: none)
  // derived, filled by finalize()
  std::vector<lm::Leaf> leaves;    // flattened, colex order
  std::vector<int> mode_leaves;    // leaves per top-level mode
  int64_t size = 1;
  int64_t cosize = 1;              // see lm_layout_cosize
};

namespace lm {

void finalize(lm_layout& L);                  // fills the derived fields
std::vector<Leaf> flatten(const Node& n);
std::vector<Node> top_modes(const lm_layout& L);
int64_t eval_affine(const std::vector<Leaf>& leaves, int64_t idx);
std::string to_string(const lm_layout& L);
std::vector<Leaf> coalesce_leaves(const std::vector<Leaf>& leaves);
bool affine_injective(std::vector<Leaf> leaves);
bool compact_bijection(const std::vector<Leaf>& leaves);
std::vector<int64_t> thread_coordinate(const lm_layout& thr, int64_t t);

// ---------------------------------------------------------------------------
// Fast division by an invariant 32-bit divisor: Granlund & Montgomery,
// "Division by invariant integers using multiplication" (PLDI 1994), the
// round-up method of their Figure 4.1.  For 1 <= d < 2^31 and any 32-bit n:
//   l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1,
//   t = mulhi(m, n), q = (t + ((n - t) >> min(l,1))) >> max(l-1, 0).
// ---------------------------------------------------------------------------
struct FastDiv {
  uint32_t d = 1, m = 1, s1 = 0, s2 = 0;
};

inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  if (d == 0) fail(LM_E_INVALID);
  uint32_t l = 0;
  while ((uint64_t(1) << l) < d) ++l;
  f.d = d;
  f.m = uint32_t(((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1);
  f.s1 = l > 0 ? 1u : 0u;
  f.s2 = l > 0 ? l - 1 : 0u;
  return f;
}

#if defined(__CUDACC__)
__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
  uint32_t t = __umulhi(f.m, n);
  return (t + ((n - t) >> f.s1)) >> f.s2;
}
#endif
inline uint32_t fdiv_host(uint32_t n, const FastDiv& f) {
  uint32_t t = uint32_t((uint64_t(f.m) * n) >> 32);
  return (t + ((n - t) >> f.s1)) >> f.s2;
}

// ---------------------------------------------------------------------------
// Kernel argument blocks (passed by value; everything in BYTES unless noted).
// ---------------------------------------------------------------------------
constexpr int kMaxModes = 8;    // joint modes of a piece after coalescing
constexpr int kMaxLeaves = 16;  // leaves of one side (GENERIC over own leaves)
constexpr int kMaxTile = 6;     // modes of a staged tile per role

struct GenericArgs {
  uint64_t n = 0;            // elements in the piece
  uint64_t i0 = 0;           // logical index of the piece's first element
  int32_t ns = 0, nd = 0;    // leaves per side
  int32_t eb = 1;            // element bytes moved per element (1..16)
  int32_t wide = 0;          // 1 if n >= 2^32 (64-bit index arithmetic)
  uint32_t s_ext[kMaxLeaves], d_ext[kMaxLeaves];
  FastDiv s_div[kMaxLeaves], d_div[kMaxLeaves];
  int64_t s_str[kMaxLeaves], d_str[kMaxLeaves];  // bytes per coordinate step
  int64_t s_ext64[kMaxLeaves], d_ext64[kMaxLeaves];
  int64_t s_base = 0, d_base = 0;                // bytes
  Swz s_swz, d_swz;                              // in bytes
};

struct VecArgs {
  uint32_t n_vec = 0;        // vectors in the piece
  int32_t nm = 0;            // modes; mode 0 counts vectors along the run
  uint32_t ext[kMaxModes];
  FastDiv div[kMaxModes];
  int64_t s[kMaxModes], d[kMaxModes];   // bytes per coordinate step
  int64_t s_base = 0, d_base = 0;       // bytes
  Swz s_swz, d_swz;                     // in bytes
  // tiled form (tiled == 1): tiles of tile_vecs vectors over the first nt
  // modes (tile extents t_ext), a grid of n_tiles tiles over the rest
  int32_t tiled = 0;
  int32_t unroll = 4;                   // vectors per thread per tile (4|8)
  uint32_t tile_vecs = 0;
  int32_t nt = 0;
  uint32_t t_ext[kMaxModes];
  FastDiv t_div[kMaxModes];
  int64_t t_s[kMaxModes], t_d[kMaxModes];
  uint32_t n_tiles = 0;
  int32_t ng = 0;
  uint32_t g_ext[kMaxModes];
  FastDiv g_pre[kMaxModes], g_div[kMaxModes];
  int64_t g_s[kMaxModes], g_d[kMaxModes];
  // in-register interleave (PATH_ZIP): each vector index names zip_rows
  // source vectors zip_s_row bytes apart and zip_rows consecutive
  // destination vectors
  int32_t zip_rows = 0;
  int64_t zip_s_row = 0;
};

struct StagedArgs {
  // tiles: colex over the grid modes
  uint32_t n_tiles = 0;
  int32_t ng = 0;
  uint32_t g_ext[kMaxModes];
  FastDiv g_pre[kMaxModes];             // division by the product of faster
  FastDiv g_div[kMaxModes];             //   grid extents, then by the extent
  int64_t g_s[kMaxModes], g_d[kMaxModes];
  int64_t s_base = 0, d_base = 0;
  Swz s_swz, d_swz;                     // global swizzles, bytes
  // load side: n_seg segments (colex over the src-outer tile modes), each
  // cps 16-byte chunks long
  uint32_t n_lchunks = 0, cps = 1;
  FastDiv cps_div;
  int32_t nso = 0;
  uint32_t so_ext[kMaxTile];
  FastDiv so_div[kMaxTile];
  int64_t so_s[kMaxTile];               // src bytes per segment coordinate
  uint32_t so_m[kMaxTile];              // smem bytes per segment coordinate
  // store side: n_dout spans (colex over the dst-outer tile modes), each cpd
  // 16-byte chunks of dst-contiguous elements
  uint32_t n_schunks = 0, cpd = 1;
  FastDiv cpd_div;
  int32_t ndo = 0;
  uint32_t do_ext[kMaxTile];
  FastDiv do_div[kMaxTile];
  int64_t do_d[kMaxTile];               // dst bytes per span coordinate
  uint32_t do_m[kMaxTile];              // smem bytes per span coordinate
  int32_t ndi = 0;                      // dst-inner modes, dst order
  uint32_t di_ext[kMaxTile];
  FastDiv di_div[kMaxTile];
  uint32_t di_m[kMaxTile];              // smem bytes per coordinate
  // transpose store (store_mode 1): micro-tiles of R rows (dst-fast mode b)
  // by one 16-byte chunk (V elements of the src-fast mode a)
  int32_t store_mode = 0;               // 0 gather, 1 transpose
  int32_t xr = 0;                       // R, rows per micro-tile
  uint32_t n_micro = 0;                 // micro-tiles per tile
  uint32_t n_bc = 1;                    // micro-tiles along b
  FastDiv bc_div;
  uint32_t n_ac = 1;                    // micro-tiles along a
  FastDiv ac_div;
  int32_t x_acfast = 0;                 // 1: micro-tile index runs along a
                                        //    first (conflict-free rows
                                        //    without a swizzle)
  uint32_t x_pitch = 0;                 // smem bytes between rows
  int32_t x_blocks = 0;                 // 1: micro-tiles in warp blocks of
                                        //    8 along b x 4 along a (each
                                        //    quarter-warp 8 bank groups of a
                                        //    128-byte-swizzled image)
  uint32_t x_region = 0;                // smem bytes per 128-byte column
                                        //    region of the tile (0: rows of
                                        //    the whole tile width)
  int64_t x_da = 0;                     // dst bytes per 16-byte chunk of a
  int64_t x_db = 0;                     // dst bytes per R rows of b
  int64_t x_vstep = 0;                  // dst bytes between output vectors
  // shared memory
  uint32_t stage_bytes = 0;
  Swz m_swz;                            // smem swizzle, bytes
  int32_t threads = 256;                // block size
  int32_t stages = 2;                   // cp.async pipeline depth (2 or 3)
  // bulk-copy form (bulk == 1): one cp.async.bulk per source segment into an
  // unswizzled image, mbarrier pipeline; needs the whole source reach
  // (src_reach bytes from the buffer start) inside the caller's capacity
  int64_t load_reach = 0;               // largest byte a tile's loads reach
                                        // past the tile origin, + 1
  int32_t bulk = 0;
  int32_t bulk_stages = 3;
  uint32_t n_seg = 0, seg_bytes = 0;
  int64_t src_reach = 0;
  // tensor-map form (tma == 1, with bulk == 1; transposes): the piece's
  // source is a tensor of t_rank dimensions -- dim 0 the unit-stride mode,
  // dim 1 the tile's other mode, then the rest -- loaded one box of t_box
  // elements per tile by a single cp.async.bulk.tensor; grid mode k
  // advances dim g_tdim[k] by g_tstep[k] elements per coordinate.  The box
  // lands densely (rows of t_box[0] elements), which is the image the
  // store side reads.
  int32_t tma = 0;
  int32_t t_swz128 = 0;                 // boxes of 128-byte rows, swizzled
                                        // (t_regions of them per tile, one
                                        // per x_region of the stage)
  uint32_t t_regions = 1;
  int32_t t_rank = 0;
  uint64_t t_dim[5];                    // extents, elements
  uint64_t t_stride[5];                 // bytes (t_stride[0] unused)
  uint32_t t_box[5];
  int32_t g_tdim[kMaxModes];
  uint32_t g_tstep[kMaxModes];
};

// Tiled copy of a pair without a common refinement (PATH_GTILE).  One side
// ("inner") runs with unit stride along the logical index; the other
// ("outer") has its unit-stride leaf at logical weight W, so with
// i = u + W*v (u < W) the outer side's offset is lo(u) + hi(v) -- its
// leaves before that leaf over u, the rest over v -- and contiguous along
// v, while the inner side's offset (its full decomposition of i) is
// contiguous along u.  Tiles of tile_u (32 or 64) x kGtV (u, v) are staged through
// shared memory: read along the source's contiguous direction, written
// along the destination's.  32-bit logical indices.
constexpr int kGtU = 32, kGtV = 64;
constexpr int kGtLeaves = 4;            // leaves per part at most
struct GTileArgs {
  uint64_t n = 0;
  uint32_t W = 1;                       // u extent
  uint32_t nv = 0;                      // v extent, n / W
  uint32_t tile_u = 32;                 // tile extent along u (32 | 64)
  uint32_t n_ut = 0, n_vt = 0;          // tiles along u and v
  FastDiv ut_div;                       // division by n_ut
  int32_t outer_src = 1;                // 1: the source is the outer side
  int32_t n_lo = 0, n_hi = 0, n_in = 0;
  uint32_t lo_ext[kMaxLeaves];
  FastDiv lo_div[kMaxLeaves];
  int64_t lo_str[kMaxLeaves];           // bytes
  uint32_t hi_ext[kMaxLeaves];
  FastDiv hi_div[kMaxLeaves];
  int64_t hi_str[kMaxLeaves];           // bytes
  uint32_t in_ext[kMaxLeaves];
  FastDiv in_div[kMaxLeaves];
  int64_t in_str[kMaxLeaves];           // bytes
  // the steps a thread takes between its elements, as digits in each part's
  // mixed radix: u by 4 over the lo leaves, the index by 8 * W over the
  // inner leaves
  uint32_t lo_step[kMaxLeaves];
  uint32_t in_step[kMaxLeaves];
  // each step's offset change (bytes): without carries the sum of its
  // digits times the strides (*_dstep), plus, per carry out of leaf k,
  // stride[k + 1] - ext[k] * stride[k] (*_cadj)
  int64_t lo_dstep = 0, in_dstep = 0;
  int64_t lo_cadj[kMaxLeaves];
  int64_t in_cadj[kMaxLeaves];
  int64_t s_base = 0, d_base = 0;       // bytes
  Swz s_swz, d_swz;                     // bytes
  int32_t narrow = 0;                   // every byte offset below 2^31
  // tensor-map form (tma == 1): an outer source that is a plain matrix --
  // v its unit-stride leaf (nv coordinates), u one leaf of t_ustride bytes
  // -- loaded one 128-byte-swizzled box of t_vpr v by tile_u u per 128-byte
  // column region (t_regions per tile); the store phase reads 16-byte
  // chunks and steps the inner digits by in_step1 (the next v) or in_jump
  // (the first v of the thread's next chunk)
  int32_t tma = 0;
  uint32_t t_regions = 0, t_vpr = 0;
  int64_t t_ustride = 0;
  uint32_t in_step1[kMaxLeaves];
  uint32_t in_jump[kMaxLeaves];
  int64_t in_dstep1 = 0, in_djump = 0;
};

struct EvalArgs {
  uint64_t n = 0;
  int32_t nl = 0;
  int32_t wide = 0;
  uint32_t ext[kMaxLeaves];
  FastDiv div[kMaxLeaves];
  int64_t ext64[kMaxLeaves];
  int64_t str[kMaxLeaves];              // elements
  Swz swz;                              // elements
  // tiled form: tiles of tile_elems consecutive indices, whose offsets are
  // inner(r) + outer(tile) -- the inner leaves (n_in) cover the first
  // leaves and part of one (tile_elems = their product), the outer leaves
  // (n_out) number the tiles
  int32_t n_in = 0, n_out = 0;
  uint32_t tile_elems = 0;
  uint64_t n_tiles = 0;
  uint32_t in_ext[kMaxLeaves];
  FastDiv in_div[kMaxLeaves];
  int64_t in_str[kMaxLeaves];
  uint32_t out_ext[kMaxLeaves];
  FastDiv out_div[kMaxLeaves];
  int64_t out_str[kMaxLeaves];
};

// ---------------------------------------------------------------------------
// The lowered plan.
// ---------------------------------------------------------------------------
enum Path : int {
  PATH_GENERIC = 0,
  PATH_VEC = 1,
  PATH_STAGED = 2,
  PATH_ZIP = 3,
  PATH_GTILE = 4
};

struct JMode {
  int64_t e, s, d;  // extent, src stride, dst stride (elements)
};

struct Piece {
  Path path = PATH_GENERIC;
  std::vector<JMode> modes;  // joint modes (empty for the non-joint case)
  int64_t s_base = 0, d_base = 0;  // elements
  int vec_bytes = 0;               // VEC: bytes per vector
  int64_t tile_elems = 0;          // STAGED: elements per tile
  int xr = 0;                      // STAGED transpose: rows per micro-tile
  GenericArgs gen;                 // always filled (fallback)
  GTileArgs gt;                    // PATH_GTILE
  VecArgs vec;
  StagedArgs st;
  int64_t bank_cost = 0, bank_ideal = 0;  // STAGED: simulated smem wavefronts
  int64_t bank_read = 0, bank_read_ideal = 0;  // of which the store side's reads
};

}  // namespace lm

struct lm_plan {
  int eb = 1;
  int64_t size = 0, src_cosize = 0, dst_cosize = 0;
  lm::Swz s_swz, d_swz;  // elements
  bool joint = true;
  std::vector<lm::Piece> pieces;
  // element ranges the copy can touch, [lo, hi): [0, cosize) unless the
  // plan is a shard (lm_plan_copy_shard) of a joint pair
  int64_t src_lo = 0, src_hi = 0, dst_lo = 0, dst_hi = 0;
  bool dst_own = true;  // no other shard writes inside [dst_lo, dst_hi)
  std::string describe;
};

// A thread-value partitioned tile copy (lm_tv.cpp plans it, lm_tv.cu runs it).
struct lm_tv_plan {
  lm_tv_args args{};
  int64_t src_cosize = 0, dst_cosize = 0;  // elements
  std::string describe;
};

namespace lm {
// Shared-memory wavefronts of one warp access (lm_plan.cpp): addr in bytes,
// `bytes` per lane.
int64_t warp_wavefronts(const int64_t* addr, const bool* valid, int bytes);
// Common refinement of two layouts' leaves into coalesced joint modes
// (lm_plan.cpp); false when the extents do not nest.
bool joint_modes(const lm_layout& src, const lm_layout& dst,
                 std::vector<JMode>& out);
int launch_tv(const lm_tv_plan& plan, const char* src, char* dst,
              void* stream);  // lm_tv.cu
// The Pitch/Strips search of lm_stripmined_tune (lm_plan.cpp); with
// `partition` only one-group maps that tile the tile.
int stripmined_search(int64_t threads, int64_t k_row, int64_t rows,
                      int64_t ld, int elem_bytes, int vec_elems,
                      const lm_layout* smem, bool partition, int64_t* pitch,
                      int64_t* strips, int64_t* segments,
                      int64_t* wavefronts);

// implemented in lm_kernels.cu
int launch_piece(const lm_plan& plan, const Piece& pc, const char* src,
                 int64_t src_cap_bytes, char* dst, void* stream);
int launch_eval(const lm_layout& L, void* table, int offset_bytes,
                void* stream);
void set_cuda_error(int e);
unsigned int* device_status_word();  // device address, current device
}  // namespace lm
