// sm_103a kernels of the layoutmove library and the ABI entry points that
// enqueue them.
//
//  layout_eval  : table[i] = L(i)                        (one offset/thread)
//  GENERIC copy : out[dst(i)] = in[src(i)], one element per thread, each
//                 side's offset from its own leaves
//  VEC copy     : the same over 16-byte vectors along the run both sides
//                 share (the common vector of the inverse layouts,
//                 "CUTE布局代数" §2.3)
//  STAGED copy  : tiles staged through shared memory -- 16-byte cp.async
//                 loads along the source's contiguous modes into an
//                 XOR-swizzled shared-memory image, double-buffered across
//                 tiles ("CUTE布局代数" §5.2), then per-element gathers into
//                 16-byte stores along the destination's contiguous modes.
//                 The thread -> chunk map is pitch-linear over the tile's
//                 chunks (the PitchLinearStripminedThreadMap article §1.2:
//                 adjacent threads take adjacent 16-byte chunks), so every
//                 warp-wide load and store covers whole 128-byte lines.
//
// No tensor cores: the work is pure data movement.

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <utility>
#include <cstring>
#include <map>
#include <mutex>

#include "lm_internal.h"
#include "lm_mbar.cuh"

namespace lm {

namespace {
thread_local int g_last_cuda = 0;
}
void set_cuda_error(int e) { g_last_cuda = e; }

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------

template <int B>
struct VecT;
template <>
struct VecT<16> {
  using T = uint4;
};
template <>
struct VecT<8> {
  using T = uint2;
};
template <>
struct VecT<4> {
  using T = uint32_t;
};
template <>
struct VecT<2> {
  using T = uint16_t;
};
template <>
struct VecT<1> {
  using T = uint8_t;
};

// Programmatic dependent launch: a kernel lets the next kernel on its stream
// start as soon as all of its own blocks are resident, and waits for the
// previous kernel to complete (and its writes to be visible) before its
// first global memory access.  Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

// Streaming global accesses: every byte is read once and written once, so
// both are marked evict-first in L1/L2.
template <class T>
__device__ __forceinline__ T ld_stream(const T* p) {
  return __ldcs(p);
}
template <class T>
__device__ __forceinline__ void st_stream(T* p, const T& v) {
  __stcs(p, v);
}

// cp.async: 16-byte copies from global to shared memory (with a source
// size, the rest zero-filled), groups and waits.
__device__ __forceinline__ void cp_async16(uint32_t smem_addr, const void* g,
                                           int src_bytes) {
  asm volatile(
      "cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_addr),
      "l"(g), "r"(src_bytes)
      : "memory");
}
__device__ __forceinline__ void cp_async16_full(uint32_t smem_addr,
                                                const void* g) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_addr),
               "l"(g)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ int64_t swz_apply(const Swz& z, int64_t o) {
  return z.b > 0 ? (o ^ ((o >> z.s) & (((int64_t(1) << z.b) - 1) << z.m))) : o;
}

__device__ __forceinline__ uint32_t swz_apply32(const Swz& z, uint32_t o) {
  return z.b > 0 ? (o ^ ((o >> z.s) & (((1u << z.b) - 1u) << z.m))) : o;
}

// offset (bytes) of a 32-bit colex index over one side's leaves
__device__ __forceinline__ int64_t side_offset32(uint32_t q, int n,
                                                 const uint32_t* ext,
                                                 const FastDiv* div,
                                                 const int64_t* str) {
  int64_t off = 0;
#pragma unroll
  for (int k = 0; k < kMaxLeaves; ++k) {
    if (k >= n) break;
    const uint32_t qn = fdiv(q, div[k]);
    off += int64_t(q - qn * ext[k]) * str[k];
    q = qn;
  }
  return off;
}

__device__ __forceinline__ int64_t side_offset64(uint64_t q, int n,
                                                 const int64_t* ext,
                                                 const int64_t* str) {
  int64_t off = 0;
  for (int k = 0; k < n; ++k) {
    const uint64_t e = uint64_t(ext[k]);
    off += int64_t(q % e) * str[k];
    q /= e;
  }
  return off;
}

// ---------------------------------------------------------------------------
// layout_eval
// ---------------------------------------------------------------------------

template <typename OUT>
__global__ void __launch_bounds__(256)
    lm_eval_kernel(const __grid_constant__ EvalArgs a, OUT* __restrict__ table) {
  pdl_trigger();
  pdl_wait();
  const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
  for (uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < a.n;
       i += stride) {
    int64_t off;
    if (a.wide) {
      off = side_offset64(i, a.nl, a.ext64, a.str);
    } else {
      off = side_offset32(uint32_t(i), a.nl, a.ext, a.div, a.str);
    }
    table[i] = OUT(swz_apply(a.swz, off));
  }
}

// The same table in 16-byte stores: when the first leaf's extent is a
// multiple of R = 16 / sizeof(OUT), each thread decomposes one index in R
// and steps the first leaf for the other R - 1 entries.
template <typename OUT>
__global__ void __launch_bounds__(256)
    lm_eval_vec_kernel(const __grid_constant__ EvalArgs a,
                       OUT* __restrict__ table) {
  constexpr int R = 16 / int(sizeof(OUT));
  pdl_trigger();
  pdl_wait();
  const uint64_t nq = a.n / R;
  const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
  for (uint64_t q = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; q < nq;
       q += stride) {
    const uint64_t i = q * R;
    const int64_t off =
        a.wide ? side_offset64(i, a.nl, a.ext64, a.str)
               : side_offset32(uint32_t(i), a.nl, a.ext, a.div, a.str);
    OUT v[R];
#pragma unroll
    for (int u = 0; u < R; ++u) v[u] = OUT(swz_apply(a.swz, off + u * a.str[0]));
    uint4 w;
    memcpy(&w, v, 16);
    __stcs(reinterpret_cast<uint4*>(table) + q, w);
  }
}

// The table tile by tile: a tile is tile_elems consecutive indices whose
// offsets split into a part inside the tile (the first leaves) and the
// tile's base (the rest).  Each thread computes the in-tile offsets of its U
// vectors once; per tile it adds the base, one decomposition of the tile
// number, and writes 16-byte vectors (a warp writes 512 contiguous bytes).
template <typename OUT, int U>
__global__ void __launch_bounds__(256)
    lm_eval_tiled_kernel(const __grid_constant__ EvalArgs a,
                         OUT* __restrict__ table) {
  constexpr int R = 16 / int(sizeof(OUT));
  const uint32_t tid = threadIdx.x, nt = blockDim.x;
  const uint32_t n_vec = a.tile_elems / R;
  int64_t off[U][R];
#pragma unroll
  for (int u = 0; u < U; ++u)
#pragma unroll
    for (int e = 0; e < R; ++e) {
      uint32_t r = (tid + uint32_t(u) * nt) * R + uint32_t(e);
      int64_t o = 0;
#pragma unroll
      for (int k = 0; k < kMaxLeaves; ++k) {
        if (k >= a.n_in) break;
        const uint32_t q = fdiv(r, a.in_div[k]);
        o += int64_t(r - q * a.in_ext[k]) * a.in_str[k];
        r = q;
      }
      off[u][e] = o;
    }
  pdl_trigger();
  pdl_wait();
  for (uint64_t tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x) {
    int64_t base = 0;
    uint32_t q = uint32_t(tile);
#pragma unroll
    for (int k = 0; k < kMaxLeaves; ++k) {
      if (k >= a.n_out) break;
      const uint32_t qn = fdiv(q, a.out_div[k]);
      base += int64_t(q - qn * a.out_ext[k]) * a.out_str[k];
      q = qn;
    }
    uint4* out = reinterpret_cast<uint4*>(table + tile * a.tile_elems);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t j = tid + uint32_t(u) * nt;
      if (j >= n_vec) break;
      OUT v[R];
#pragma unroll
      for (int e = 0; e < R; ++e) v[e] = OUT(swz_apply(a.swz, base + off[u][e]));
      uint4 w;
      memcpy(&w, v, 16);
      __stcs(out + j, w);
    }
  }
}

// ---------------------------------------------------------------------------
// GENERIC copy
// ---------------------------------------------------------------------------

template <int EB>
__global__ void __launch_bounds__(256)
    lm_generic_kernel(const __grid_constant__ GenericArgs a,
                      const char* __restrict__ src, char* __restrict__ dst) {
  using T = typename VecT<EB>::T;
  pdl_trigger();
  pdl_wait();
  const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
  for (uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < a.n;
       i += stride) {
    int64_t so, dof;
    const uint64_t ig = i + a.i0;
    if (a.wide) {
      so = side_offset64(ig, a.ns, a.s_ext64, a.s_str);
      dof = side_offset64(ig, a.nd, a.d_ext64, a.d_str);
    } else {
      so = side_offset32(uint32_t(ig), a.ns, a.s_ext, a.s_div, a.s_str);
      dof = side_offset32(uint32_t(ig), a.nd, a.d_ext, a.d_div, a.d_str);
    }
    so = swz_apply(a.s_swz, a.s_base + so);
    dof = swz_apply(a.d_swz, a.d_base + dof);
    *reinterpret_cast<T*>(dst + dof) =
        *reinterpret_cast<const T*>(src + so);
  }
}

// ---------------------------------------------------------------------------
// GTILE copy: a pair without a common refinement, tile by tile through
// shared memory (GTileArgs)
// ---------------------------------------------------------------------------

// offset (bytes) of a 32-bit index over n leaves
__device__ __forceinline__ int64_t leaves_offset(uint32_t q, int n,
                                                 const uint32_t* ext,
                                                 const FastDiv* div,
                                                 const int64_t* str) {
  int64_t off = 0;
#pragma unroll
  for (int k = 0; k < kMaxLeaves; ++k) {
    if (k >= n) break;
    const uint32_t qn = fdiv(q, div[k]);
    off += int64_t(q - qn * ext[k]) * str[k];
    q = qn;
  }
  return off;
}

// A position in the mixed radix of up to NL leaves, with its byte
// offset: set once by division, then advanced by a constant step given as
// digits (add with carries), so a thread's next element costs a few adds.
template <int NL, typename OFF>
struct Digits {
  uint32_t c[NL];
  OFF off;

  __device__ __forceinline__ void set(uint32_t q, int n, const uint32_t* ext,
                                      const FastDiv* div, const int64_t* str) {
    off = 0;
#pragma unroll
    for (int k = 0; k < NL; ++k) {
      c[k] = 0;
      if (k < n) {
        const uint32_t qn = fdiv(q, div[k]);
        c[k] = q - qn * ext[k];
        off += OFF(c[k]) * OFF(str[k]);
        q = qn;
      }
    }
  }
  // Add the step whose digits are d.  The offset changes by dsum (the
  // digits times the strides) plus cadj[k] per carry out of leaf k
  // (stride[k + 1] - ext[k] * stride[k]), both computed on the host.  The
  // last leaf may run past its extent: the step never leaves the caller's
  // range, so no carry out of it is ever needed, and its digit is not kept.
  __device__ __forceinline__ void step(int n, const uint32_t* ext,
                                       const uint32_t* d, int64_t dsum,
                                       const int64_t* cadj) {
    uint32_t carry = 0;
    OFF delta = OFF(dsum);
#pragma unroll
    for (int k = 0; k + 1 < NL; ++k) {
      if (k + 1 < n) {
        uint32_t x = c[k] + d[k] + carry;
        carry = x >= ext[k] ? 1u : 0u;
        if (carry) {
          x -= ext[k];
          delta += OFF(cadj[k]);
        }
        c[k] = x;
      }
    }
    off += delta;
  }
};

// One element from global into shared memory: cp.async for 4, 8 and 16
// bytes (asynchronous: the caller commits and waits), a plain load and
// store otherwise.
template <int EB>
__device__ __forceinline__ void elem_to_shared(void* s, const char* g) {
  if constexpr (EB >= 4) {
    const uint32_t a = uint32_t(__cvta_generic_to_shared(s));
    if constexpr (EB == 16)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(a),
                   "l"(g)
                   : "memory");
    else
      asm volatile("cp.async.ca.shared.global [%0], [%1], %2;\n" ::"r"(a),
                   "l"(g), "n"(EB)
                   : "memory");
  } else {
    using T = typename VecT<EB>::T;
    *reinterpret_cast<T*>(s) = *reinterpret_cast<const T*>(g);
  }
}

// OUTER_SRC: the source is the outer side -- it is read along v (lanes
// over v, its offset lo(u) + hi(v)) and the destination, the inner side,
// written along u (lanes over u, its offset from the full index).  The
// other way round otherwise.  Two shared tiles of TU x (kGtV + 1)
// elements (the pad keeps the lanes that walk along u in distinct banks):
// a block's next tile loads (cp.async) while it stores the current one.
template <int EB, bool OUTER_SRC, int NL, typename OFF, int TU>
__global__ void __launch_bounds__(256)
    lm_gtile_kernel(const __grid_constant__ GTileArgs a,
                    const char* __restrict__ src, char* __restrict__ dst) {
  using T = typename VecT<EB>::T;
  constexpr int RU = 256 / kGtV;  // rows of u per pass, lanes over v
  constexpr int CV = 256 / TU;    // columns of v per pass, lanes over u
  extern __shared__ __align__(16) unsigned char gt_smem[];
  typedef T Tile[TU][kGtV + 1];
  Tile* tiles = reinterpret_cast<Tile*>(gt_smem);
  pdl_trigger();
  pdl_wait();
  const uint32_t t = threadIdx.x;
  const uint32_t n_tiles = a.n_ut * a.n_vt;
  const uint32_t vl_v = t % kGtV, ul_v = t / kGtV;
  const uint32_t ul_u = t % TU, vl_u = t / TU;
  // swizzles only where a side has one (a uniform test, not per element)
  const bool sswz = a.s_swz.b > 0, dswz = a.d_swz.b > 0;
  auto sw_s = [&](OFF o) {
    return sswz ? OFF(swz_apply(a.s_swz, int64_t(o))) : o;
  };
  auto sw_d = [&](OFF o) {
    return dswz ? OFF(swz_apply(a.d_swz, int64_t(o))) : o;
  };
  auto origin = [&](uint32_t ti, uint32_t* u0, uint32_t* v0) {
    const uint32_t vt = fdiv(ti, a.ut_div);
    *u0 = (ti - vt * a.n_ut) * TU;
    *v0 = vt * kGtV;
  };
  auto load = [&](uint32_t ti, Tile& tl) {
    uint32_t u0, v0;
    origin(ti, &u0, &v0);
    if constexpr (OUTER_SRC) {  // the outer source along v
      const uint32_t v = v0 + vl_v;
      if (v >= a.nv) return;
      const OFF base = OFF(
          a.s_base + leaves_offset(v, a.n_hi, a.hi_ext, a.hi_div, a.hi_str));
      Digits<NL, OFF> lo;
      lo.set(u0 + ul_v, a.n_lo, a.lo_ext, a.lo_div, a.lo_str);
#pragma unroll
      for (int p = 0; p < TU / RU; ++p) {
        const uint32_t ul = ul_v + uint32_t(RU * p);
        if (u0 + ul >= a.W) break;
        if (p) lo.step(a.n_lo, a.lo_ext, a.lo_step, a.lo_dstep, a.lo_cadj);
        elem_to_shared<EB>(&tl[ul][vl_v],
                           src + sw_s(base + lo.off));
      }
    } else {  // the inner source along u
      const uint32_t u = u0 + ul_u;
      if (u >= a.W) return;
      Digits<NL, OFF> in;
      in.set(u + a.W * (v0 + vl_u), a.n_in, a.in_ext, a.in_div, a.in_str);
#pragma unroll
      for (int p = 0; p < kGtV / CV; ++p) {
        const uint32_t vl = vl_u + uint32_t(CV * p);
        if (v0 + vl >= a.nv) break;
        if (p) in.step(a.n_in, a.in_ext, a.in_step, a.in_dstep, a.in_cadj);
        elem_to_shared<EB>(&tl[ul_u][vl],
                           src + sw_s(OFF(a.s_base) + in.off));
      }
    }
  };
  auto store = [&](uint32_t ti, const Tile& tl) {
    uint32_t u0, v0;
    origin(ti, &u0, &v0);
    if constexpr (OUTER_SRC) {  // the inner destination along u
      const uint32_t u = u0 + ul_u;
      if (u >= a.W) return;
      Digits<NL, OFF> in;
      in.set(u + a.W * (v0 + vl_u), a.n_in, a.in_ext, a.in_div, a.in_str);
#pragma unroll
      for (int p = 0; p < kGtV / CV; ++p) {
        const uint32_t vl = vl_u + uint32_t(CV * p);
        if (v0 + vl >= a.nv) break;
        if (p) in.step(a.n_in, a.in_ext, a.in_step, a.in_dstep, a.in_cadj);
        *reinterpret_cast<T*>(dst + sw_d(OFF(a.d_base) + in.off)) =
            tl[ul_u][vl];
      }
    } else {  // the outer destination along v
      const uint32_t v = v0 + vl_v;
      if (v >= a.nv) return;
      const OFF base = OFF(
          a.d_base + leaves_offset(v, a.n_hi, a.hi_ext, a.hi_div, a.hi_str));
      Digits<NL, OFF> lo;
      lo.set(u0 + ul_v, a.n_lo, a.lo_ext, a.lo_div, a.lo_str);
#pragma unroll
      for (int p = 0; p < TU / RU; ++p) {
        const uint32_t ul = ul_v + uint32_t(RU * p);
        if (u0 + ul >= a.W) break;
        if (p) lo.step(a.n_lo, a.lo_ext, a.lo_step, a.lo_dstep, a.lo_cadj);
        *reinterpret_cast<T*>(dst + sw_d(base + lo.off)) =
            tl[ul][vl_v];
      }
    }
  };
  uint32_t ti = blockIdx.x;
  if (ti >= n_tiles) return;
  load(ti, tiles[0]);
  cp_async_commit();
  for (int buf = 0;; buf ^= 1) {
    const uint32_t next = ti + gridDim.x;
    // the other tile was last read before the barrier ending the previous
    // iteration
    if (next < n_tiles) load(next, tiles[buf ^ 1]);
    cp_async_commit();
    cp_async_wait<1>();  // this tile's copies have landed
    __syncthreads();
    store(ti, tiles[buf]);
    __syncthreads();
    if (next >= n_tiles) break;
    ti = next;
  }
  cp_async_wait<0>();
}

// ---------------------------------------------------------------------------
// VEC copy: 16-byte (or narrower) vectors along the shared run
// ---------------------------------------------------------------------------

constexpr int kVecUnroll = 4;

template <int VB>
__global__ void __launch_bounds__(256)
    lm_vec_kernel(const __grid_constant__ VecArgs a,
                  const char* __restrict__ src, char* __restrict__ dst) {
  using T = typename VecT<VB>::T;
  pdl_trigger();
  pdl_wait();
  const uint64_t nthreads = uint64_t(gridDim.x) * blockDim.x;
  for (uint64_t q0 = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
       q0 < a.n_vec; q0 += kVecUnroll * nthreads) {
    T v[kVecUnroll];
    int64_t doff[kVecUnroll];
#pragma unroll
    for (int u = 0; u < kVecUnroll; ++u) {
      const uint64_t q64 = q0 + u * nthreads;
      doff[u] = -1;
      if (q64 < a.n_vec) {
        uint32_t q = uint32_t(q64);
        int64_t s = a.s_base, d = a.d_base;
#pragma unroll
        for (int k = 0; k < kMaxModes; ++k) {
          if (k >= a.nm) break;
          const uint32_t qn = fdiv(q, a.div[k]);
          const int64_t c = int64_t(q - qn * a.ext[k]);
          s += c * a.s[k];
          d += c * a.d[k];
          q = qn;
        }
        s = swz_apply(a.s_swz, s);
        doff[u] = swz_apply(a.d_swz, d);
        v[u] = ld_stream(reinterpret_cast<const T*>(src + s));
      }
    }
#pragma unroll
    for (int u = 0; u < kVecUnroll; ++u)
      if (doff[u] >= 0) st_stream(reinterpret_cast<T*>(dst + doff[u]), v[u]);
  }
}

// Tile origin offsets (bytes) over a grid of ng modes.  Lane k of each group
// of 8 lanes computes grid coordinate k in parallel (tile / product of the
// faster extents, mod the extent); a 3-step butterfly of warp shuffles sums
// the contributions, so every lane of the warp ends with both totals.
__device__ __forceinline__ void grid_base(int ng, const uint32_t* ext,
                                          const FastDiv* pre,
                                          const FastDiv* div,
                                          const int64_t* gs, const int64_t* gd,
                                          uint32_t tile, int64_t& sb,
                                          int64_t& db) {
  const int k = threadIdx.x & 7;
  int64_t s = 0, d = 0;
  if (k < ng) {
    uint32_t c = fdiv(tile, pre[k]);
    c -= fdiv(c, div[k]) * ext[k];
    s = int64_t(c) * gs[k];
    d = int64_t(c) * gd[k];
  }
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, off);
    d += __shfl_xor_sync(0xffffffffu, d, off);
  }
  sb = s;
  db = d;
}

// VEC, tiled: each thread owns U vectors of a tile (the same
// offsets in every tile, computed once); the next tile's vectors are loaded
// into registers before the current tile's are stored.
template <int VB, int U>
__global__ void __launch_bounds__(256)
    lm_vec_tiled_kernel(const __grid_constant__ VecArgs a,
                        const char* __restrict__ src, char* __restrict__ dst) {
  using T = typename VecT<VB>::T;
  const uint32_t tid = threadIdx.x, nt = blockDim.x;
  int32_t so[U], dof[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    uint32_t j = tid + uint32_t(u) * nt;
    so[u] = -1;
    dof[u] = 0;
    if (j < a.tile_vecs) {
      int64_t s = 0, d = 0;
#pragma unroll
      for (int k = 0; k < kMaxModes; ++k) {
        if (k >= a.nt) break;
        const uint32_t jn = fdiv(j, a.t_div[k]);
        const int64_t c = int64_t(j - jn * a.t_ext[k]);
        s += c * a.t_s[k];
        d += c * a.t_d[k];
        j = jn;
      }
      so[u] = int32_t(s);
      dof[u] = int32_t(d);
    }
  }
  pdl_trigger();
  pdl_wait();
  uint32_t tile = blockIdx.x;
  if (tile >= a.n_tiles) return;
  int64_t sb, db;
  grid_base(a.ng, a.g_ext, a.g_pre, a.g_div, a.g_s, a.g_d, tile, sb, db);
  T cur[U];
#pragma unroll
  for (int u = 0; u < U; ++u)
    if (so[u] >= 0)
      cur[u] = ld_stream(reinterpret_cast<const T*>(
          src + swz_apply(a.s_swz, a.s_base + sb + so[u])));
  for (;;) {
    const uint64_t next64 = uint64_t(tile) + gridDim.x;
    const bool has_next = next64 < a.n_tiles;
    T nxt[U];
    int64_t nsb = 0, ndb = 0;
    if (has_next) {
      grid_base(a.ng, a.g_ext, a.g_pre, a.g_div, a.g_s, a.g_d,
                uint32_t(next64), nsb, ndb);
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (so[u] >= 0)
          nxt[u] = ld_stream(reinterpret_cast<const T*>(
              src + swz_apply(a.s_swz, a.s_base + nsb + so[u])));
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (so[u] >= 0)
        st_stream(reinterpret_cast<T*>(
                   dst + swz_apply(a.d_swz, a.d_base + db + dof[u])),
               cur[u]);
    if (!has_next) break;
#pragma unroll
    for (int u = 0; u < U; ++u) cur[u] = nxt[u];
    tile = uint32_t(next64);
    db = ndb;
  }
}

// ---------------------------------------------------------------------------
// STAGED copy
//
// The load side is shared: each thread owns a fixed set of 16-byte chunks of
// the tile's source image (the same for every tile) and moves them with
// cp.async into a swizzled shared-memory image, one tile ahead of the store
// side (two stages).  The store side is a policy:
//   GatherStore : per-element gathers from shared memory into 16-byte
//                 destination vectors (any tile structure);
//   XposeStore  : micro-tiles of R rows x 16 bytes read with 16-byte shared
//                 loads and transposed in registers (byte permutes), for
//                 tiles that are a 2-D transpose.
// ---------------------------------------------------------------------------


__device__ __forceinline__ uint4 lds128(const unsigned char* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// Tile origin offsets (bytes).  Lane k of each group of 8 lanes computes
// grid coordinate k in parallel (tile / product-of-faster-extents, mod the
// extent); a 3-step butterfly of warp shuffles sums the contributions, so
// every lane of the warp ends with both totals.
__device__ __forceinline__ void tile_base(const StagedArgs& a, uint32_t tile,
                                          int64_t& sb, int64_t& db) {
  const int k = threadIdx.x & 7;
  int64_t s = 0, d = 0;
  if (k < a.ng) {
    uint32_t c = fdiv(tile, a.g_pre[k]);
    c -= fdiv(c, a.g_div[k]) * a.g_ext[k];
    s = int64_t(c) * a.g_s[k];
    d = int64_t(c) * a.g_d[k];
  }
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, off);
    d += __shfl_xor_sync(0xffffffffu, d, off);
  }
  sb = s;
  db = d;
}

template <int L>
struct LoadSlots {
  int32_t src[L];
  uint32_t sm[L];

  __device__ __forceinline__ void init(const StagedArgs& a, uint32_t tid,
                                       uint32_t nt) {
#pragma unroll
    for (int k = 0; k < L; ++k) {
      const uint32_t j = tid + uint32_t(k) * nt;
      src[k] = -1;
      sm[k] = 0;
      if (j < a.n_lchunks) {
        const uint32_t seg = fdiv(j, a.cps_div);
        const uint32_t c = j - seg * a.cps;
        int64_t srel = int64_t(c) * 16;
        uint32_t mrel = c * 16u;
        uint32_t r = seg;
#pragma unroll
        for (int t = 0; t < kMaxTile; ++t) {
          if (t >= a.nso) break;
          const uint32_t rn = fdiv(r, a.so_div[t]);
          const uint32_t x = r - rn * a.so_ext[t];
          srel += int64_t(x) * a.so_s[t];
          mrel += x * a.so_m[t];
          r = rn;
        }
        src[k] = int32_t(srel);
        sm[k] = swz_apply32(a.m_swz, mrel);
      }
    }
  }

  __device__ __forceinline__ void issue(const StagedArgs& a, const char* src_p,
                                        int64_t src_cap, int64_t base,
                                        uint32_t sm_stage) const {
    if (a.s_swz.b == 0 && base + a.load_reach <= src_cap) {
      // common case: no source swizzle, the whole tile inside the buffer
      const char* p = src_p + base;
#pragma unroll
      for (int k = 0; k < L; ++k)
        if (src[k] >= 0) cp_async16_full(sm_stage + sm[k], p + src[k]);
      return;
    }
#pragma unroll
    for (int k = 0; k < L; ++k) {
      if (src[k] < 0) continue;
      const int64_t off = swz_apply(a.s_swz, base + src[k]);
      const int64_t room = src_cap - off;
      const int nbytes = room >= 16 ? 16 : (room > 0 ? int(room) : 0);
      cp_async16(sm_stage + sm[k], nbytes ? src_p + off : src_p, nbytes);
    }
  }
};

template <int EB>
struct GatherStore {
  static constexpr int kLoadSlots = EB >= 8 ? 8 : 4;
  static constexpr int V = 16 / EB;
  static constexpr int MaxS = (16 / V) < 1 ? 1 : ((16 / V) > 4 ? 4 : 16 / V);
  int32_t dst[MaxS];
  uint32_t sm[MaxS][V];

  __device__ __forceinline__ void init(const StagedArgs& a, uint32_t tid,
                                       uint32_t nt) {
#pragma unroll
    for (int k = 0; k < MaxS; ++k) {
      const uint32_t j = tid + uint32_t(k) * nt;
      dst[k] = -1;
#pragma unroll
      for (int e = 0; e < V; ++e) sm[k][e] = 0;
      if (j < a.n_schunks) {
        const uint32_t o = fdiv(j, a.cpd_div);
        const uint32_t p = j - o * a.cpd;
        int64_t drel = int64_t(p) * 16;
        uint32_t mb = 0, r = o;
#pragma unroll
        for (int t = 0; t < kMaxTile; ++t) {
          if (t >= a.ndo) break;
          const uint32_t rn = fdiv(r, a.do_div[t]);
          const uint32_t x = r - rn * a.do_ext[t];
          drel += int64_t(x) * a.do_d[t];
          mb += x * a.do_m[t];
          r = rn;
        }
        dst[k] = int32_t(drel);
#pragma unroll
        for (int e = 0; e < V; ++e) {
          uint32_t q = p * uint32_t(V) + uint32_t(e);
          uint32_t m = mb;
#pragma unroll
          for (int t = 0; t < kMaxTile; ++t) {
            if (t >= a.ndi) break;
            const uint32_t qn = fdiv(q, a.di_div[t]);
            m += (q - qn * a.di_ext[t]) * a.di_m[t];
            q = qn;
          }
          sm[k][e] = swz_apply32(a.m_swz, m);
        }
      }
    }
  }

  __device__ __forceinline__ void store(const StagedArgs& a,
                                        const unsigned char* smst, char* dst_p,
                                        int64_t dbase) const {
#pragma unroll
    for (int k = 0; k < MaxS; ++k) {
      if (dst[k] < 0) continue;
      uint32_t w[4];
      if constexpr (EB == 16) {
        const uint4 v = lds128(smst + sm[k][0]);
        w[0] = v.x;
        w[1] = v.y;
        w[2] = v.z;
        w[3] = v.w;
      } else if constexpr (EB == 8) {
        const uint2 x = *reinterpret_cast<const uint2*>(smst + sm[k][0]);
        const uint2 y = *reinterpret_cast<const uint2*>(smst + sm[k][1]);
        w[0] = x.x;
        w[1] = x.y;
        w[2] = y.x;
        w[3] = y.y;
      } else if constexpr (EB == 4) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          w[e] = *reinterpret_cast<const uint32_t*>(smst + sm[k][e]);
      } else if constexpr (EB == 2) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t lo = *reinterpret_cast<const uint16_t*>(smst + sm[k][2 * i]);
          const uint32_t hi = *reinterpret_cast<const uint16_t*>(smst + sm[k][2 * i + 1]);
          w[i] = __byte_perm(lo, hi, 0x5410);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t b0 = smst[sm[k][4 * i]];
          const uint32_t b1 = smst[sm[k][4 * i + 1]];
          const uint32_t b2 = smst[sm[k][4 * i + 2]];
          const uint32_t b3 = smst[sm[k][4 * i + 3]];
          w[i] = __byte_perm(__byte_perm(b0, b1, 0x0040),
                             __byte_perm(b2, b3, 0x0040), 0x5410);
        }
      }
      const int64_t off =
          a.d_swz.b ? swz_apply(a.d_swz, dbase + dst[k]) : dbase + dst[k];
      st_stream(reinterpret_cast<uint4*>(dst_p + off),
                make_uint4(w[0], w[1], w[2], w[3]));
    }
  }
};

// Register transpose of R rows of V = 16/EB elements: output word W of the
// column-by-column order (element f = in[f % R][f / R]).  W is a
// compile-time constant after unrolling, so every index is too.
template <int EB, int R>
__device__ __forceinline__ uint32_t xword(const uint32_t (&in)[R][4], int W) {
  if constexpr (EB == 4) {
    return in[W % R][W / R];
  } else if constexpr (EB == 8) {
    const int f = W / 2;
    return in[f % R][(f / R) * 2 + (W % 2)];
  } else if constexpr (EB == 2) {
    const int f0 = 2 * W, f1 = 2 * W + 1;
    const int a0 = f0 / R, b0 = f0 % R, a1 = f1 / R, b1 = f1 % R;
    const uint32_t sel =
        ((a0 & 1) ? 0x32u : 0x10u) | ((a1 & 1) ? 0x7600u : 0x5400u);
    return __byte_perm(in[b0][a0 / 2], in[b1][a1 / 2], sel);
  } else {  // EB == 1
    uint32_t t[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int f0 = 4 * W + 2 * h, f1 = f0 + 1;
      const int a0 = f0 / R, b0 = f0 % R, a1 = f1 / R, b1 = f1 % R;
      const uint32_t sel = uint32_t(a0 % 4) | (uint32_t(4 + a1 % 4) << 4);
      t[h] = __byte_perm(in[b0][a0 / 4], in[b1][a1 / 4], sel);
    }
    return __byte_perm(t[0], t[1], 0x5410);
  }
}

// ---------------------------------------------------------------------------
// ZIP copy: interleave of R source rows without shared memory.  Vector q of
// the piece names R source vectors (rows zip_s_row bytes apart, the same
// 16-byte column) and R consecutive destination vectors; the R x V block is
// transposed in registers.  A warp's loads of one row and its stores are
// both contiguous.
// ---------------------------------------------------------------------------

template <int EB, int R, int U>
__global__ void __launch_bounds__(256)
    lm_zip_kernel(const __grid_constant__ VecArgs a,
                  const char* __restrict__ src, char* __restrict__ dst) {
  pdl_trigger();
  pdl_wait();
  const uint64_t nthreads = uint64_t(gridDim.x) * blockDim.x;
  for (uint64_t q0 = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
       q0 < a.n_vec; q0 += U * nthreads) {
    uint32_t in[U][R][4];
    int64_t doff[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint64_t q64 = q0 + u * nthreads;
      doff[u] = -1;
      if (q64 < a.n_vec) {
        uint32_t q = uint32_t(q64);
        int64_t s = a.s_base, d = a.d_base;
#pragma unroll
        for (int k = 0; k < kMaxModes; ++k) {
          if (k >= a.nm) break;
          const uint32_t qn = fdiv(q, a.div[k]);
          const int64_t c = int64_t(q - qn * a.ext[k]);
          s += c * a.s[k];
          d += c * a.d[k];
          q = qn;
        }
        doff[u] = d;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint4 v =
              ld_stream(reinterpret_cast<const uint4*>(src + s + r * a.zip_s_row));
          in[u][r][0] = v.x;
          in[u][r][1] = v.y;
          in[u][r][2] = v.z;
          in[u][r][3] = v.w;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (doff[u] < 0) continue;
#pragma unroll
      for (int j = 0; j < R; ++j)
        st_stream(reinterpret_cast<uint4*>(dst + doff[u] + 16 * j),
                  make_uint4(xword<EB, R>(in[u], 4 * j),
                             xword<EB, R>(in[u], 4 * j + 1),
                             xword<EB, R>(in[u], 4 * j + 2),
                             xword<EB, R>(in[u], 4 * j + 3)));
    }
  }
}

template <int EB, int R>
struct XposeStore {
  static constexpr int kLoadSlots = R >= 8 ? 8 : 4;
  static constexpr int MaxM = R >= 8 ? 1 : 2;
  int32_t dst[MaxM];
  uint32_t sm[MaxM][R];  // swizzled smem address of each row's chunk

  __device__ __forceinline__ void init(const StagedArgs& a, uint32_t tid,
                                       uint32_t nt) {
#pragma unroll
    for (int k = 0; k < MaxM; ++k) {
      const uint32_t j = tid + uint32_t(k) * nt;
      dst[k] = -1;
#pragma unroll
      for (int r = 0; r < R; ++r) sm[k][r] = 0;
      if (j < a.n_micro) {
        uint32_t ac, bc;
        if (a.x_blocks) {
          // warp blocks of 8 micro-tiles along b by 4 along a; each
          // quarter-warp covers 8 bank groups of the swizzled image
          const uint32_t w = j >> 5, l = j & 31, nwb = a.n_bc >> 3;
          const uint32_t wa = w / nwb, wb = w - wa * nwb;
          if constexpr (R == 4) {
            bc = 8u * wb + 2u * (l >> 3) + (l & 1u);
            ac = 4u * wa + ((l >> 1) & 3u);
          } else {
            bc = 8u * wb + 4u * ((l >> 3) & 1u) + (l & 3u);
            ac = 4u * wa + 2u * (l >> 4) + ((l >> 2) & 1u);
          }
        } else if (a.x_acfast) {
          bc = fdiv(j, a.ac_div);
          ac = j - bc * a.n_ac;
        } else {
          ac = fdiv(j, a.bc_div);
          bc = j - ac * a.n_bc;
        }
        dst[k] = int32_t(int64_t(ac) * a.x_da + int64_t(bc) * a.x_db);
        // chunk ac of the row: in its 128-byte column region when the tile
        // is stored as such regions
        const uint32_t col = a.x_region ? (ac >> 3) * a.x_region + (ac & 7u) * 16u
                                        : ac * 16u;
        const uint32_t lin = bc * uint32_t(R) * a.x_pitch + col;
#pragma unroll
        for (int r = 0; r < R; ++r)
          sm[k][r] = swz_apply32(a.m_swz, lin + uint32_t(r) * a.x_pitch);
      }
    }
  }

  __device__ __forceinline__ void store(const StagedArgs& a,
                                        const unsigned char* smst, char* dst_p,
                                        int64_t dbase) const {
    const int32_t vstep = int32_t(a.x_vstep);
#pragma unroll
    for (int k = 0; k < MaxM; ++k) {
      if (dst[k] < 0) continue;
      uint32_t in[R][4];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const uint4 v = lds128(smst + sm[k][r]);
        in[r][0] = v.x;
        in[r][1] = v.y;
        in[r][2] = v.z;
        in[r][3] = v.w;
      }
      if (a.d_swz.b == 0) {
        char* p = dst_p + (dbase + dst[k]);
#pragma unroll
        for (int j = 0; j < R; ++j)
          st_stream(reinterpret_cast<uint4*>(p + j * vstep),
                    make_uint4(xword<EB, R>(in, 4 * j),
                               xword<EB, R>(in, 4 * j + 1),
                               xword<EB, R>(in, 4 * j + 2),
                               xword<EB, R>(in, 4 * j + 3)));
      } else {
        const int64_t base = dbase + dst[k];
#pragma unroll
        for (int j = 0; j < R; ++j) {
          const int64_t off = swz_apply(a.d_swz, base + j * vstep);
          st_stream(reinterpret_cast<uint4*>(dst_p + off),
                    make_uint4(xword<EB, R>(in, 4 * j),
                               xword<EB, R>(in, 4 * j + 1),
                               xword<EB, R>(in, 4 * j + 2),
                               xword<EB, R>(in, 4 * j + 3)));
        }
      }
    }
  }
};

// NS-stage pipeline: the loads of the NS-1 tiles after the current one are
// in flight while the current tile is stored.  Every iteration commits one
// cp.async group (possibly empty), so waiting until at most NS-1 groups are
// pending means the current tile's group has landed.
template <int EB, class Store, int NS>
__global__ void __launch_bounds__(256)
    lm_staged_kernel(const __grid_constant__ StagedArgs a,
                     const char* __restrict__ src, char* __restrict__ dst,
                     int64_t src_cap) {
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t tid = threadIdx.x;
  const uint32_t nt = blockDim.x;
  LoadSlots<Store::kLoadSlots> ls;
  ls.init(a, tid, nt);
  Store st;
  st.init(a, tid, nt);
  pdl_trigger();
  pdl_wait();

  uint64_t tile = blockIdx.x;
  if (tile >= a.n_tiles) return;
  const uint64_t G = gridDim.x;
  const uint32_t smem0 = uint32_t(__cvta_generic_to_shared(smem));
  int64_t dq[NS];  // dst bases of the tiles in flight, oldest first
#pragma unroll
  for (int i = 0; i < NS - 1; ++i) {
    const uint64_t t = tile + uint64_t(i) * G;
    dq[i] = 0;
    if (t < a.n_tiles) {
      int64_t sb;
      tile_base(a, uint32_t(t), sb, dq[i]);
      ls.issue(a, src, src_cap, a.s_base + sb,
               smem0 + uint32_t(i) * a.stage_bytes);
    }
    cp_async_commit();
  }
  int stage = 0;
  for (;;) {
    const uint64_t ahead = tile + uint64_t(NS - 1) * G;
    dq[NS - 1] = 0;
    if (ahead < a.n_tiles) {
      int64_t sb;
      tile_base(a, uint32_t(ahead), sb, dq[NS - 1]);
      const int s_ahead = (stage + NS - 1) % NS;
      ls.issue(a, src, src_cap, a.s_base + sb,
               smem0 + uint32_t(s_ahead) * a.stage_bytes);
    }
    cp_async_commit();
    cp_async_wait<NS - 1>();
    __syncthreads();
    st.store(a, smem + size_t(stage) * a.stage_bytes, dst, a.d_base + dq[0]);
    __syncthreads();
    tile += G;
    if (tile >= a.n_tiles) break;
    stage = (stage + 1) % NS;
#pragma unroll
    for (int i = 0; i < NS - 1; ++i) dq[i] = dq[i + 1];
  }
  cp_async_wait<0>();
}

// ---------------------------------------------------------------------------
// STAGED copy, bulk-copy form
//
// Warp 0 is the producer: per tile it announces the tile's byte count on the
// stage's "full" mbarrier and its lanes issue one cp.async.bulk per source
// segment (row) straight into the stage's padded shared-memory image.  Every
// warp consumes: it waits on "full", runs the store policy on the stage and
// arrives on the stage's "empty" mbarrier, which the producer waits on before
// refilling the stage NS tiles later.  No block-wide barrier sits in the
// tile loop.
//
// Every wait is bounded (kWaitCycles of clock64, about a second): a wait
// that gives up sets bit 0 of g_lm_device_status, and the producer then
// waits for the copies it still has in flight (kDrainCycles per stage) so
// that the block leaves no bulk copy writing into shared memory it no longer
// owns.  The drain is bounded too: copies from global memory complete unless
// the memory system itself has failed, so a drain that still runs out sets
// bit 1 -- the block has exited with copies in flight, which may overwrite
// the shared memory of a block that runs on that SM later -- and the host
// must then treat the device's results as suspect.  The host reads the word
// with lm_device_status.
// ---------------------------------------------------------------------------

__device__ unsigned int g_lm_device_status = 0;
constexpr int kBulkSegsPerLane = 4;  // up to 128 segments per tile


__device__ __forceinline__ void bulk_g2s(uint32_t dst_smem, const void* src,
                                         uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];\n" ::"r"(dst_smem),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// One box of a tiled tensor map into shared memory (the tensor-memory-
// accelerator copy), completing on an mbarrier; c[] are the box's first
// element coordinates, dim 0 first.
__device__ __forceinline__ void tma_g2s(uint32_t dst_smem, const CUtensorMap* m,
                                        int rank, int32_t c0, int32_t c1,
                                        int32_t c2, int32_t c3, int32_t c4,
                                        uint32_t bar) {
  const uint64_t map = reinterpret_cast<uint64_t>(m);
  const int32_t c[5] = {c0, c1, c2, c3, c4};
  switch (rank) {
    case 2:
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::"
          "complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst_smem),
          "l"(map), "r"(c[0]), "r"(c[1]), "r"(bar)
          : "memory");
      break;
    case 3:
      asm volatile(
          "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::"
          "complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(
              dst_smem),
          "l"(map), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(bar)
          : "memory");
      break;
    case 4:
      asm volatile(
          "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::"
          "complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];\n" ::"r"(
              dst_smem),
          "l"(map), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(bar)
          : "memory");
      break;
    default:
      asm volatile(
          "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::"
          "complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];\n" ::"r"(
              dst_smem),
          "l"(map), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(c[4]),
          "r"(bar)
          : "memory");
      break;
  }
}

// Bytes of dynamic shared memory a bulk-form block asks for: mbarriers
// (128 bytes), the stages, and slack to align them (128 bytes, or 1024 for
// tensor-map stages).
inline int bulk_smem_bytes(const StagedArgs& a, int ns) {
  return int((a.tma ? 128 + 1024 : 256) + ns * a.stage_bytes);
}

// The bulk-copy STAGED kernel.  TMA == false: one cp.async.bulk per source
// segment; TMA == true: one tensor-map box per tile (tmap describes the
// piece's source, StagedArgs::tma).
template <int EB, class Store, int NS, bool TMA>
__global__ void __launch_bounds__(256)
    lm_bulk_kernel(const __grid_constant__ StagedArgs a,
                   const __grid_constant__ CUtensorMap tmap,
                   const char* __restrict__ src, char* __restrict__ dst) {
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t tid = threadIdx.x, nt = blockDim.x;
  const uint32_t warp = tid >> 5, lane = tid & 31, n_warps = nt >> 5;
  // mbarriers from the first 128-byte boundary, stages from the next
  // 1024-byte one (swizzled tensor copies need 1024-byte aligned
  // destinations, plain ones 128; the launch adds the slack)
  const uint32_t base = uint32_t(__cvta_generic_to_shared(smem));
  const uint32_t bars = (base + 127u) & ~127u;
  auto full = [&](uint32_t s) { return bars + 8u * s; };
  auto empty = [&](uint32_t s) { return bars + 8u * (NS + s); };
  const uint32_t stage0 =
      TMA ? ((bars + 128u + 1023u) & ~1023u) : bars + 128u;
  unsigned char* stages = smem + (stage0 - base);

  Store st;
  st.init(a, tid, nt);
  // producer slots: segments lane, lane + 32, ... (source and smem offsets)
  int32_t seg_src[kBulkSegsPerLane];
  uint32_t seg_sm[kBulkSegsPerLane];
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < kBulkSegsPerLane; ++k) {
      const uint32_t g = lane + 32u * uint32_t(k);
      seg_src[k] = -1;
      seg_sm[k] = 0;
      if (g < a.n_seg) {
        int64_t srel = 0;
        uint32_t mrel = 0, r = g;
#pragma unroll
        for (int t = 0; t < kMaxTile; ++t) {
          if (t >= a.nso) break;
          const uint32_t rn = fdiv(r, a.so_div[t]);
          const uint32_t x = r - rn * a.so_ext[t];
          srel += int64_t(x) * a.so_s[t];
          mrel += x * a.so_m[t];
          r = rn;
        }
        seg_src[k] = int32_t(srel);
        seg_sm[k] = mrel;
      }
    }
  }
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), n_warps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();

  if (blockIdx.x >= a.n_tiles) return;
  const uint32_t G = gridDim.x;
  const uint32_t n_local = (a.n_tiles - blockIdx.x + G - 1) / G;
  const uint32_t tile_bytes = a.n_seg * a.seg_bytes;
  bool ok = true;
  uint32_t issued = 0;  // tiles the producer has issued

  // producer: tile number i of this block into stage i % NS
  auto issue = [&](uint32_t i) -> bool {
    const uint32_t s = i % NS;
    if (i >= uint32_t(NS) && !warp_wait(empty(s), ((i / NS) - 1) & 1))
      return false;
    const uint32_t sdst = stage0 + s * a.stage_bytes;
    if constexpr (TMA) {
      if (lane == 0) {
        // the tile's box origin: grid coordinates times the box steps
        int32_t c0 = 0, c1 = 0, c2 = 0, c3 = 0, c4 = 0;
        uint32_t t = blockIdx.x + i * G;
#pragma unroll
        for (int k = 0; k < kMaxModes; ++k) {
          if (k >= a.ng) break;
          const uint32_t q = fdiv(t, a.g_div[k]);
          const int32_t v = int32_t((t - q * a.g_ext[k]) * a.g_tstep[k]);
          const int32_t d = a.g_tdim[k];
          c0 += d == 0 ? v : 0;
          c1 += d == 1 ? v : 0;
          c2 += d == 2 ? v : 0;
          c3 += d == 3 ? v : 0;
          c4 += d == 4 ? v : 0;
          t = q;
        }
        mbar_arrive_expect_tx(full(s), tile_bytes);
        // one box per 128-byte column region (one box when unswizzled)
        for (uint32_t g = 0; g < a.t_regions; ++g)
          tma_g2s(sdst + g * a.x_region, &tmap, a.t_rank,
                  c0 + int32_t(g * a.t_box[0]), c1, c2, c3, c4, full(s));
      }
      __syncwarp();
    } else {
      int64_t sb, db;
      tile_base(a, blockIdx.x + i * G, sb, db);
      if (lane == 0) mbar_arrive_expect_tx(full(s), tile_bytes);
      __syncwarp();
      const char* base = src + a.s_base + sb;
#pragma unroll
      for (int k = 0; k < kBulkSegsPerLane; ++k)
        if (seg_src[k] >= 0)
          bulk_g2s(sdst + seg_sm[k], base + seg_src[k], a.seg_bytes, full(s));
    }
    return true;
  };

  if (warp == 0)
    for (uint32_t i = 0; i < uint32_t(NS - 1) && i < n_local && ok; ++i) {
      ok = issue(i);
      issued += ok ? 1u : 0u;
    }
  uint32_t i = 0;
  for (; i < n_local; ++i) {
    if (warp == 0 && ok && i + NS - 1 < n_local) {
      ok = issue(i + NS - 1);
      issued += ok ? 1u : 0u;
    }
    const uint32_t s = i % NS;
    if (!ok || !warp_wait(full(s), (i / NS) & 1)) {
      ok = false;
      break;
    }
    int64_t sb, db;
    tile_base(a, blockIdx.x + i * G, sb, db);
    st.store(a, stages + size_t(s) * a.stage_bytes, dst, a.d_base + db);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(s));
  }
  if (!ok) {
    if (lane == 0) atomicOr(&g_lm_device_status, 1u);
    if (warp == 0) {  // drain this block's copies still in flight
      bool drained = true;
      for (uint32_t j = i; j < issued && drained; ++j)
        drained = warp_wait(full(j % NS), (j / NS) & 1, kDrainCycles);
      if (!drained && lane == 0) atomicOr(&g_lm_device_status, 2u);
    }
  }
}

// ---------------------------------------------------------------------------
// GTILE with tensor-map loads (GTileArgs::tma): the outer source is a plain
// matrix, each 64 x 64 (u, v) tile arrives as 128-byte-swizzled boxes (one
// per 128-byte column region: element chunk c of row u at chunk c ^ (u % 8))
// issued by one thread, two tiles in flight on mbarriers.  Each thread then
// reads 16-byte chunks of one row u -- 8 consecutive rows, one chunk
// column, hit 8 distinct bank groups -- and writes their elements along u
// into the inner destination, stepping its digits.  Every wait is bounded;
// the block votes on the outcome, so it leaves together, and a timeout
// drains the copies in flight as the bulk kernels do.
// ---------------------------------------------------------------------------

template <int EB, typename OFF>
__global__ void __launch_bounds__(256)
    lm_gtma_kernel(const __grid_constant__ GTileArgs a,
                   const __grid_constant__ CUtensorMap tmap,
                   char* __restrict__ dst) {
  using T = typename VecT<EB>::T;
  constexpr int TU = 64;
  constexpr int VPC = 16 / EB;             // v per 16-byte chunk
  constexpr int CP = 256 / TU;             // chunk columns a pass spans
  constexpr int PER = kGtV / VPC / CP;     // chunks per thread per tile
  constexpr uint32_t REGION = TU * 128;    // bytes of one column region
  constexpr uint32_t STAGE = uint32_t(kGtV) * EB * TU;
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t base = uint32_t(__cvta_generic_to_shared(smem));
  const uint32_t bar = (base + 127u) & ~127u;  // two mbarriers
  const uint32_t st0 = (bar + 128u + 1023u) & ~1023u;
  const unsigned char* stages = smem + (st0 - base);
  const uint32_t t = threadIdx.x;
  if (t == 0) {
    mbar_init(bar, 1);
    mbar_init(bar + 8, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();
  const uint32_t n_tiles = a.n_ut * a.n_vt;
  uint32_t ti = blockIdx.x;
  if (ti >= n_tiles) return;
  const uint32_t G = gridDim.x;
  const uint32_t ul = t % TU, cl = t / TU;
  const bool dswz = a.d_swz.b > 0;
  auto origin = [&](uint32_t tile, uint32_t* u0, uint32_t* v0) {
    const uint32_t vt = fdiv(tile, a.ut_div);
    *u0 = (tile - vt * a.n_ut) * TU;
    *v0 = vt * kGtV;
  };
  auto issue = [&](uint32_t tile, uint32_t s) {  // thread 0
    uint32_t u0, v0;
    origin(tile, &u0, &v0);
    mbar_arrive_expect_tx(bar + 8u * s, STAGE);
    for (uint32_t r = 0; r < a.t_regions; ++r)
      tma_g2s(st0 + s * STAGE + r * REGION, &tmap, 2,
              int32_t(v0 + r * a.t_vpr), int32_t(u0), 0, 0, 0, bar + 8u * s);
  };
  if (t == 0) issue(ti, 0);
  bool ok = true;
  uint32_t i = 0, next = 0;
  for (;; ++i) {
    const uint32_t s = i & 1u;
    next = ti + G;
    // stage s ^ 1 held the tile before, released by the last vote
    if (t == 0 && next < n_tiles) issue(next, s ^ 1u);
    ok = mbar_wait(bar + 8u * s, (i >> 1) & 1u);
    if (ok) {
      uint32_t u0, v0;
      origin(ti, &u0, &v0);
      const uint32_t u = u0 + ul;
      if (u < a.W) {
        const unsigned char* row = stages + s * STAGE + ul * 128u;
        Digits<2, OFF> in;
        in.set(u + a.W * (v0 + cl * VPC), a.n_in, a.in_ext, a.in_div,
               a.in_str);
        in.off += OFF(a.d_base);
#pragma unroll
        for (int k = 0; k < PER; ++k) {
          const uint32_t ch = cl + uint32_t(CP * k);
          const uint32_t vf = v0 + ch * VPC;
          if (vf >= a.nv) break;
          if (k)
            in.step(a.n_in, a.in_ext, a.in_jump, a.in_djump, a.in_cadj);
          const uint4 w = *reinterpret_cast<const uint4*>(
              row + (ch >> 3) * REGION + (((ch & 7u) ^ (ul & 7u)) << 4));
          T vals[VPC];
          memcpy(vals, &w, 16);
          const bool whole = vf + uint32_t(VPC) <= a.nv;
#pragma unroll
          for (int e = 0; e < VPC; ++e) {
            if (!whole && vf + uint32_t(e) >= a.nv) break;
            if (e)
              in.step(a.n_in, a.in_ext, a.in_step1, a.in_dstep1,
                      a.in_cadj);
            const OFF o = in.off;
            *reinterpret_cast<T*>(
                dst + (dswz ? OFF(swz_apply(a.d_swz, int64_t(o))) : o)) =
                vals[e];
          }
        }
      }
    }
    ok = __syncthreads_and(ok);
    if (!ok || next >= n_tiles) break;
    ti = next;
  }
  if (!ok && t == 0) {
    atomicOr(&g_lm_device_status, 1u);
    // drain this block's boxes still in flight: tile i's, and the next
    // one's if it was issued
    bool drained = mbar_wait(bar + 8u * (i & 1u), (i >> 1) & 1u, kDrainCycles);
    if (drained && next < n_tiles)
      drained = mbar_wait(bar + 8u * ((i + 1) & 1u), ((i + 1) >> 1) & 1u,
                          kDrainCycles);
    if (!drained) atomicOr(&g_lm_device_status, 2u);
  }
}

// Self-test of the bounded wait: one warp waits on an mbarrier that, with
// arrive == 0, nothing ever arrives at.  The wait gives up after kWaitCycles
// and records the timeout exactly as the copy kernels do.
__global__ void lm_selftest_wait_kernel(int arrive) {
  __shared__ __align__(8) unsigned long long bar;
  const uint32_t b = uint32_t(__cvta_generic_to_shared(&bar));
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  if (arrive && threadIdx.x == 0) mbar_arrive(b);
  const bool ok = warp_wait(b, 0);
  if (!ok && threadIdx.x == 0) atomicOr(&g_lm_device_status, 1u);
}

// ---------------------------------------------------------------------------
// host side: launches
// ---------------------------------------------------------------------------

// Device address of g_lm_device_status on the current device (looked up
// once per device), for kernels of other files that record timeouts.
unsigned int* device_status_word() {
  static std::mutex mu;
  static unsigned int* addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return nullptr;
  std::lock_guard<std::mutex> g(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_lm_device_status) != cudaSuccess)
      return nullptr;
    addr[dev] = static_cast<unsigned int*>(p);
  }
  return addr[dev];
}

struct DeviceInfo {
  int sms = 0;
};

DeviceInfo device_info() {
  static std::mutex mu;
  static DeviceInfo cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return {148};
  std::lock_guard<std::mutex> g(mu);
  if (!cache[dev].sms) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    cache[dev].sms = v > 0 ? v : 148;
  }
  return cache[dev];
}

// Blocks launched: several waves beat one persistent wave (measured on
// GB300): blocks that finish are replaced at once, so the memory system
// stays busy to the end.  VEC grids are LM_WAVES_VEC (default 8) times the
// resident blocks.
uint64_t env_waves(const char* name, uint64_t dflt) {
  const char* e = std::getenv(name);
  const long long w = e ? std::atoll(e) : (long long)dflt;
  return uint64_t(w < 1 ? 1 : w);
}
uint64_t waves_vec() {
  static uint64_t v = env_waves("LM_WAVES_VEC", 8);
  return v;
}
// STAGED grids give each block about this many tiles (LM_TILES_PER_BLOCK):
// enough for the two-stage pipeline to overlap a tile's loads with the
// previous tile's stores, few enough that blocks turn over often.
uint64_t tiles_per_block() {
  static uint64_t v = env_waves("LM_TILES_PER_BLOCK", 2);
  return v;
}
uint64_t staged_grid(uint64_t n_tiles, uint64_t resident) {
  const uint64_t want = (n_tiles + tiles_per_block() - 1) / tiles_per_block();
  return std::max<uint64_t>(1, std::min<uint64_t>(want, resident * 64));
}

bool pdl_enabled() {
  static bool v = [] {
    const char* e = std::getenv("LM_PDL");
    return !(e && e[0] == '0');
  }();
  return v;
}

// Launch with the programmatic-stream-serialization attribute (see
// pdl_wait); LM_PDL=0 launches plainly.
template <typename... Params, typename... Args>
cudaError_t launch_k(void (*kern)(Params...), unsigned grid, unsigned block,
                     size_t smem, cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

int check_launch() {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_cuda_error(int(e));
    return LM_E_CUDA;
  }
  return LM_OK;
}

template <int EB>
int launch_generic_t(const GenericArgs& g, const char* src, char* dst,
                     cudaStream_t st) {
  const DeviceInfo di = device_info();
  const uint64_t want = (g.n + 255) / 256;
  const uint64_t cap = uint64_t(di.sms) * 16;
  const unsigned grid = unsigned(std::max<uint64_t>(1, std::min(want, cap)));
  launch_k(lm_generic_kernel<EB>, grid, 256, 0, st, g, src, dst);
  return check_launch();
}

int launch_generic(const GenericArgs& g0, const char* src, char* dst,
                   cudaStream_t st) {
  const uintptr_t ps = reinterpret_cast<uintptr_t>(src);
  const uintptr_t pd = reinterpret_cast<uintptr_t>(dst);
  GenericArgs g = g0;
  if ((ps | pd) % uintptr_t(g.eb)) {
    // pointers aligned to less than an element: move bytes, with one more
    // leaf (the byte inside the element) in front of each side
    if (g.ns + 1 > kMaxLeaves || g.nd + 1 > kMaxLeaves) {
      set_cuda_error(0);
      return LM_E_INVALID;
    }
    auto shift = [&](uint32_t* ext, FastDiv* div, int64_t* str,
                     int64_t* ext64, int32_t& n) {
      for (int k = n; k > 0; --k) {
        ext[k] = ext[k - 1];
        div[k] = div[k - 1];
        str[k] = str[k - 1];
        ext64[k] = ext64[k - 1];
      }
      ext[0] = uint32_t(g.eb);
      div[0] = make_fastdiv(uint32_t(g.eb));
      str[0] = 1;
      ext64[0] = g.eb;
      ++n;
    };
    shift(g.s_ext, g.s_div, g.s_str, g.s_ext64, g.ns);
    shift(g.d_ext, g.d_div, g.d_str, g.d_ext64, g.nd);
    g.n *= uint64_t(g.eb);
    g.i0 *= uint64_t(g.eb);
    if (g.n + g.i0 >= (uint64_t(1) << 31)) g.wide = 1;
    g.eb = 1;
  }
  switch (g.eb) {
    case 1: return launch_generic_t<1>(g, src, dst, st);
    case 2: return launch_generic_t<2>(g, src, dst, st);
    case 4: return launch_generic_t<4>(g, src, dst, st);
    case 8: return launch_generic_t<8>(g, src, dst, st);
    case 16: return launch_generic_t<16>(g, src, dst, st);
    default: return LM_E_INVALID;
  }
}

template <int VB, int U>
int launch_vec_tiled(const VecArgs& v, const char* src, char* dst,
                     cudaStream_t st) {
  const DeviceInfo di = device_info();
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &per_sm, lm_vec_tiled_kernel<VB, U>, 256, 0) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const uint64_t cap = uint64_t(di.sms) * uint64_t(per_sm) * waves_vec();
  const unsigned grid =
      unsigned(std::max<uint64_t>(1, std::min<uint64_t>(v.n_tiles, cap)));
  launch_k(lm_vec_tiled_kernel<VB, U>, grid, 256, 0, st, v, src, dst);
  return check_launch();
}

// Blocks in flight per vector of each thread: LM_ZIP_UNROLL (1 or 2).
int zip_unroll() {
  static const int u = [] {
    const char* e = std::getenv("LM_ZIP_UNROLL");
    return e && e[0] == '2' ? 2 : 1;
  }();
  return u;
}

template <int EB, int R, int U>
int launch_zip_u(const VecArgs& v, const char* src, char* dst,
                 cudaStream_t st) {
  const DeviceInfo di = device_info();
  const uint64_t want = (uint64_t(v.n_vec) + 256 * U - 1) / (256 * U);
  const uint64_t cap = uint64_t(di.sms) * 8 * uint64_t(waves_vec());
  const unsigned grid = unsigned(std::max<uint64_t>(1, std::min(want, cap)));
  launch_k(lm_zip_kernel<EB, R, U>, grid, 256, 0, st, v, src, dst);
  return check_launch();
}

template <int EB, int R>
int launch_zip_t(const VecArgs& v, const char* src, char* dst,
                 cudaStream_t st) {
  return zip_unroll() == 2 ? launch_zip_u<EB, R, 2>(v, src, dst, st)
                           : launch_zip_u<EB, R, 1>(v, src, dst, st);
}

int launch_zip(const VecArgs& v, int eb, const char* src, char* dst,
               cudaStream_t st) {
  switch (eb * 100 + v.zip_rows) {
    case 402: return launch_zip_t<4, 2>(v, src, dst, st);
    case 202: return launch_zip_t<2, 2>(v, src, dst, st);
    case 204: return launch_zip_t<2, 4>(v, src, dst, st);
    case 102: return launch_zip_t<1, 2>(v, src, dst, st);
    case 104: return launch_zip_t<1, 4>(v, src, dst, st);
    case 108: return launch_zip_t<1, 8>(v, src, dst, st);
    default: return LM_E_INVALID;
  }
}

template <int VB>
int launch_vec_t(const VecArgs& v, const char* src, char* dst,
                 cudaStream_t st) {
  const DeviceInfo di = device_info();
  if (v.tiled) {
    if (v.unroll == 8) return launch_vec_tiled<VB, 8>(v, src, dst, st);
    return launch_vec_tiled<VB, 4>(v, src, dst, st);
  }
  const uint64_t want = (uint64_t(v.n_vec) + 256 * kVecUnroll - 1) /
                        (256 * kVecUnroll);
  const uint64_t cap = uint64_t(di.sms) * 8;
  const unsigned grid = unsigned(std::max<uint64_t>(1, std::min(want, cap)));
  launch_k(lm_vec_kernel<VB>, grid, 256, 0, st, v, src, dst);
  return check_launch();
}

template <int EB, class Store, int NS>
int launch_staged_ns(const StagedArgs& a, const char* src, int64_t src_cap,
                     char* dst, cudaStream_t st) {
  // NS stages of at most 48 KiB / NS each: within the default 48 KiB of
  // dynamic shared memory, so no per-device attribute is needed
  const int smem = int(NS * a.stage_bytes);
  const DeviceInfo di = device_info();
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &per_sm, lm_staged_kernel<EB, Store, NS>, a.threads,
          size_t(smem)) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const unsigned grid = unsigned(
      staged_grid(a.n_tiles, uint64_t(di.sms) * uint64_t(per_sm)));
  launch_k(lm_staged_kernel<EB, Store, NS>, grid, unsigned(a.threads),
           size_t(smem), st, a, src, dst, src_cap);
  return check_launch();
}

// Dynamic shared memory above 48 KiB needs an opt-in per device and kernel
// (cached per device and kernel address).
template <typename K>
bool allow_smem(K kern, int bytes) {
  if (bytes <= 49152) return true;
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, int> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const auto key = std::make_pair(dev, reinterpret_cast<const void*>(kern));
  std::lock_guard<std::mutex> g(mu);
  auto it = done.find(key);
  if (it == done.end() || it->second < bytes) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bytes) != cudaSuccess)
      return false;
    done[key] = bytes;
  }
  return true;
}

// cuTensorMapEncodeTiled from the driver, found once through the runtime
// (the library links no driver library of its own).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType,
                                   cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// The tensor map of a piece's source (StagedArgs::tma) at `src`.
bool encode_source_map(const StagedArgs& a, int eb, const char* src,
                       CUtensorMap* m) {
  const EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const CUtensorMapDataType dt =
      eb == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
      : eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
      : eb == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32
                : CU_TENSOR_MAP_DATA_TYPE_UINT64;
  cuuint64_t dims[5], strides[4];
  cuuint32_t box[5], es[5];
  for (int k = 0; k < a.t_rank; ++k) {
    dims[k] = a.t_dim[k];
    box[k] = a.t_box[k];
    es[k] = 1;
    if (k > 0) strides[k - 1] = a.t_stride[k];
  }
  return fn(m, dt, cuuint32_t(a.t_rank),
            const_cast<char*>(src) + a.s_base, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            a.t_swz128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int EB, class Store, int NS, bool TMA>
int launch_bulk_ns(const StagedArgs& a, const char* src, char* dst,
                   cudaStream_t st) {
  const int smem = bulk_smem_bytes(a, NS);
  auto kern = lm_bulk_kernel<EB, Store, NS, TMA>;
  if (!allow_smem(kern, smem)) return LM_E_CUDA;
  CUtensorMap m;
  std::memset(&m, 0, sizeof(m));
  if constexpr (TMA) {
    if (!encode_source_map(a, EB, src, &m)) {
      set_cuda_error(0);
      return LM_E_CUDA;
    }
  }
  const DeviceInfo di = device_info();
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &per_sm, kern, a.threads, size_t(smem)) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const unsigned grid = unsigned(
      staged_grid(a.n_tiles, uint64_t(di.sms) * uint64_t(per_sm)));
  launch_k(kern, grid, unsigned(a.threads), size_t(smem), st, a, m, src, dst);
  return check_launch();
}

template <int EB, class Store, bool TMA>
int launch_bulk_t(const StagedArgs& a, const char* src, char* dst,
                  cudaStream_t st) {
  switch (a.bulk_stages) {
    case 2: return launch_bulk_ns<EB, Store, 2, TMA>(a, src, dst, st);
    case 4: return launch_bulk_ns<EB, Store, 4, TMA>(a, src, dst, st);
    default: return launch_bulk_ns<EB, Store, 3, TMA>(a, src, dst, st);
  }
}

template <int EB, class Store>
int launch_staged_t(const StagedArgs& a, const char* src, int64_t src_cap,
                    char* dst, cudaStream_t st) {
  if (a.bulk && src_cap >= a.src_reach) {
    if (a.tma && encode_tiled())
      return launch_bulk_t<EB, Store, true>(a, src, dst, st);
    return launch_bulk_t<EB, Store, false>(a, src, dst, st);
  }
  if (a.stages == 3 && 3 * a.stage_bytes <= 49152)
    return launch_staged_ns<EB, Store, 3>(a, src, src_cap, dst, st);
  return launch_staged_ns<EB, Store, 2>(a, src, src_cap, dst, st);
}

template <int EB>
int launch_xpose(const StagedArgs& a, const char* src, int64_t cap, char* dst,
                 cudaStream_t st) {
  constexpr int V = 16 / EB;
  switch (a.xr) {
    case 2:
      if constexpr (V >= 2)
        return launch_staged_t<EB, XposeStore<EB, 2>>(a, src, cap, dst, st);
      break;
    case 4:
      if constexpr (V >= 4)
        return launch_staged_t<EB, XposeStore<EB, 4>>(a, src, cap, dst, st);
      break;
    case 8:
      if constexpr (V >= 8)
        return launch_staged_t<EB, XposeStore<EB, 8>>(a, src, cap, dst, st);
      break;
    case 16:
      if constexpr (V >= 16)
        return launch_staged_t<EB, XposeStore<EB, 16>>(a, src, cap, dst, st);
      break;
    default:
      break;
  }
  return LM_E_INVALID;
}

int launch_staged(const StagedArgs& a, int eb, const char* src, int64_t cap,
                  char* dst, cudaStream_t st) {
  if (a.store_mode == 1) {
    switch (eb) {
      case 1: return launch_xpose<1>(a, src, cap, dst, st);
      case 2: return launch_xpose<2>(a, src, cap, dst, st);
      case 4: return launch_xpose<4>(a, src, cap, dst, st);
      case 8: return launch_xpose<8>(a, src, cap, dst, st);
      default: return LM_E_INVALID;
    }
  }
  switch (eb) {
    case 1: return launch_staged_t<1, GatherStore<1>>(a, src, cap, dst, st);
    case 2: return launch_staged_t<2, GatherStore<2>>(a, src, cap, dst, st);
    case 4: return launch_staged_t<4, GatherStore<4>>(a, src, cap, dst, st);
    case 8: return launch_staged_t<8, GatherStore<8>>(a, src, cap, dst, st);
    case 16: return launch_staged_t<16, GatherStore<16>>(a, src, cap, dst, st);
    default: return LM_E_INVALID;
  }
}

template <int EB, bool OUTER_SRC, int NL, typename OFF, int TU>
int launch_gtile_t(const GTileArgs& g, const char* src, char* dst,
                   cudaStream_t st) {
  auto kern = lm_gtile_kernel<EB, OUTER_SRC, NL, OFF, TU>;
  const int smem = 2 * TU * (kGtV + 1) * EB;
  if (!allow_smem(kern, smem)) return LM_E_CUDA;
  const DeviceInfo di = device_info();
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256,
                                                    size_t(smem)) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  // about two tiles per block, as for STAGED tiles
  const uint64_t tiles = uint64_t(g.n_ut) * g.n_vt;
  const unsigned grid = unsigned(std::max<uint64_t>(
      1, std::min<uint64_t>((tiles + 1) / 2,
                            uint64_t(di.sms) * uint64_t(per_sm) * 64)));
  launch_k(kern, grid, 256, size_t(smem), st, g, src, dst);
  return check_launch();
}

// kernels unrolled for 2 leaves per part with 32-bit offsets (the common
// case), else for 4 leaves with 64-bit offsets
template <int EB, int NL, typename OFF, int TU>
int launch_gtile_u(const GTileArgs& g, const char* src, char* dst,
                   cudaStream_t st) {
  return g.outer_src ? launch_gtile_t<EB, true, NL, OFF, TU>(g, src, dst, st)
                     : launch_gtile_t<EB, false, NL, OFF, TU>(g, src, dst, st);
}

template <int EB, int NL, typename OFF>
int launch_gtile_n(const GTileArgs& g, const char* src, char* dst,
                   cudaStream_t st) {
  return g.tile_u == 64 ? launch_gtile_u<EB, NL, OFF, 64>(g, src, dst, st)
                        : launch_gtile_u<EB, NL, OFF, 32>(g, src, dst, st);
}

// The tensor map of a GTILE outer source: dims (v, u), 128-byte swizzled
// boxes of t_vpr x 64.
bool encode_gtile_map(const GTileArgs& g, int eb, const char* src,
                      CUtensorMap* m) {
  const EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const CUtensorMapDataType dt = eb == 2   ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                 : eb == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32
                                           : CU_TENSOR_MAP_DATA_TYPE_UINT64;
  const cuuint64_t dims[2] = {g.nv, g.W};
  const cuuint64_t strides[1] = {cuuint64_t(g.t_ustride)};
  const cuuint32_t box[2] = {g.t_vpr, 64};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<char*>(src) + g.s_base, dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int EB, typename OFF>
int launch_gtma_t(const GTileArgs& g, const char* src, char* dst,
                  cudaStream_t st) {
  auto kern = lm_gtma_kernel<EB, OFF>;
  const int smem = 128 + 1024 + 2 * kGtV * EB * 64;
  if (!allow_smem(kern, smem)) return LM_E_CUDA;
  CUtensorMap m;
  if (!encode_gtile_map(g, EB, src, &m)) {
    set_cuda_error(0);
    return LM_E_CUDA;
  }
  const DeviceInfo di = device_info();
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256,
                                                    size_t(smem)) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const uint64_t tiles = uint64_t(g.n_ut) * g.n_vt;
  const unsigned grid = unsigned(std::max<uint64_t>(
      1, std::min<uint64_t>((tiles + 1) / 2,
                            uint64_t(di.sms) * uint64_t(per_sm) * 64)));
  launch_k(kern, grid, 256, size_t(smem), st, g, m, dst);
  return check_launch();
}

template <int EB>
int launch_gtile_e(const GTileArgs& g, const char* src, char* dst,
                   cudaStream_t st) {
  if constexpr (EB == 2 || EB == 4 || EB == 8) {
    // tensor-map loads need a 16-byte aligned source
    if (g.tma && reinterpret_cast<uintptr_t>(src + g.s_base) % 16 == 0 &&
        encode_tiled())
      return g.narrow ? launch_gtma_t<EB, int32_t>(g, src, dst, st)
                      : launch_gtma_t<EB, int64_t>(g, src, dst, st);
  }
  if (g.narrow && g.n_lo <= 2 && g.n_in <= 2)
    return launch_gtile_n<EB, 2, int32_t>(g, src, dst, st);
  return launch_gtile_n<EB, kGtLeaves, int64_t>(g, src, dst, st);
}

int launch_gtile(const GTileArgs& g, int eb, const char* src, char* dst,
                 cudaStream_t st) {
  switch (eb) {
    case 1: return launch_gtile_e<1>(g, src, dst, st);
    case 2: return launch_gtile_e<2>(g, src, dst, st);
    case 4: return launch_gtile_e<4>(g, src, dst, st);
    case 8: return launch_gtile_e<8>(g, src, dst, st);
    case 16: return launch_gtile_e<16>(g, src, dst, st);
    default: return LM_E_INVALID;
  }
}

int launch_piece(const lm_plan& P, const Piece& pc, const char* src,
                 int64_t src_cap_bytes, char* dst, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const uintptr_t ps = reinterpret_cast<uintptr_t>(src);
  const uintptr_t pd = reinterpret_cast<uintptr_t>(dst);
  if (pc.path == PATH_VEC && ((ps | pd) % uintptr_t(pc.vec_bytes)) == 0) {
    switch (pc.vec_bytes) {
      case 16: return launch_vec_t<16>(pc.vec, src, dst, st);
      case 8: return launch_vec_t<8>(pc.vec, src, dst, st);
      case 4: return launch_vec_t<4>(pc.vec, src, dst, st);
      default: break;
    }
  }
  if (pc.path == PATH_STAGED && ((ps | pd) % 16) == 0)
    return launch_staged(pc.st, P.eb, src, src_cap_bytes, dst, st);
  if (pc.path == PATH_ZIP && ((ps | pd) % 16) == 0)
    return launch_zip(pc.vec, P.eb, src, dst, st);
  if (pc.path == PATH_GTILE && ((ps | pd) % uintptr_t(P.eb)) == 0)
    return launch_gtile(pc.gt, P.eb, src, dst, st);
  return launch_generic(pc.gen, src, dst, st);
}

// Tiles for lm_eval_tiled_kernel: the largest tile of at most 2048 * R
// consecutive indices (at least 64 * R) that is the product of the first
// leaves and a divisor of the next, a multiple of R, with fewer than 2^32
// tiles and in-tile offsets in 32-bit index arithmetic.  False when none.
bool eval_tiles(const std::vector<Leaf>& c, int R, EvalArgs& a) {
  if (a.nl == 0 || a.n % uint64_t(R)) return false;
  const int64_t tmax = 2048 * int64_t(R), tmin = 64 * int64_t(R);
  int64_t best = 0;
  int best_k = -1;
  int64_t best_f = 1, before = 1;
  for (int k = 0; k < int(c.size()) && before <= tmax; ++k) {
    for (int64_t f = 1; f <= c[size_t(k)].e && before * f <= tmax; ++f) {
      if (c[size_t(k)].e % f) continue;
      const int64_t t = before * f;
      if (t % R == 0 && t > best) {
        best = t;
        best_k = k;
        best_f = f;
      }
    }
    before *= c[size_t(k)].e;
  }
  if (best < tmin || uint64_t(best) > a.n) return false;
  const uint64_t tiles = a.n / uint64_t(best);
  if (tiles >= (uint64_t(1) << 32)) return false;
  int n_in = 0, n_out = 0;
  for (int k = 0; k < int(c.size()); ++k) {
    const Leaf& l = c[size_t(k)];
    if (k < best_k || (k == best_k && best_f == l.e)) {
      a.in_ext[n_in] = uint32_t(l.e);
      a.in_str[n_in++] = l.d;
    } else if (k == best_k) {
      if (best_f > 1) {
        a.in_ext[n_in] = uint32_t(best_f);
        a.in_str[n_in++] = l.d;
      }
      a.out_ext[n_out] = uint32_t(l.e / best_f);
      a.out_str[n_out++] = mul_chk(l.d, best_f);
    } else {
      if (l.e >= (int64_t(1) << 32)) return false;
      a.out_ext[n_out] = uint32_t(l.e);
      a.out_str[n_out++] = l.d;
    }
    if (n_in > kMaxLeaves || n_out > kMaxLeaves) return false;
  }
  for (int k = 0; k < n_in; ++k) a.in_div[k] = make_fastdiv(a.in_ext[k]);
  for (int k = 0; k < n_out; ++k) a.out_div[k] = make_fastdiv(a.out_ext[k]);
  a.n_in = n_in;
  a.n_out = n_out;
  a.tile_elems = uint32_t(best);
  a.n_tiles = tiles;
  return true;
}

int launch_eval(const lm_layout& L, void* table, int offset_bytes,
                void* stream) {
  EvalArgs a;
  a.n = uint64_t(L.size);
  std::vector<Leaf> c = coalesce_leaves(L.leaves);
  if (c.size() > size_t(kMaxLeaves)) return LM_E_NOT_REPRESENTABLE;
  a.nl = int32_t(c.size());
  a.wide = L.size >= (int64_t(1) << 31) ? 1 : 0;
  for (size_t k = 0; k < c.size(); ++k) {
    a.ext64[k] = c[k].e;
    if (c[k].e >= (int64_t(1) << 31)) a.wide = 1;
    a.ext[k] = uint32_t(std::min<int64_t>(c[k].e, 0x7fffffff));
    a.div[k] = make_fastdiv(a.ext[k] ? a.ext[k] : 1u);
    a.str[k] = c[k].d;
  }
  a.swz = L.swz;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const DeviceInfo di = device_info();
  const uint64_t want = (a.n + 255) / 256;
  const unsigned grid = unsigned(
      std::max<uint64_t>(1, std::min<uint64_t>(want, uint64_t(di.sms) * 16)));
  const int R = 16 / offset_bytes;
  if (reinterpret_cast<uintptr_t>(table) % 16 == 0 && eval_tiles(c, R, a)) {
    const uint64_t per_block = 8;   // tiles per block: blocks turn over often
    const unsigned gridt = unsigned(std::max<uint64_t>(
        1, std::min<uint64_t>((a.n_tiles + per_block - 1) / per_block,
                              uint64_t(di.sms) * 64)));
    const uint32_t vecs = a.tile_elems / uint32_t(R);
    if (offset_bytes == 4) {
      if (vecs <= 4 * 256)
        launch_k(lm_eval_tiled_kernel<int32_t, 4>, gridt, 256, 0, st, a,
                 static_cast<int32_t*>(table));
      else
        launch_k(lm_eval_tiled_kernel<int32_t, 8>, gridt, 256, 0, st, a,
                 static_cast<int32_t*>(table));
    } else {
      if (vecs <= 4 * 256)
        launch_k(lm_eval_tiled_kernel<int64_t, 4>, gridt, 256, 0, st, a,
                 static_cast<int64_t*>(table));
      else
        launch_k(lm_eval_tiled_kernel<int64_t, 8>, gridt, 256, 0, st, a,
                 static_cast<int64_t*>(table));
    }
    return check_launch();
  }
  if (a.nl > 0 && c[0].e % R == 0 &&
      reinterpret_cast<uintptr_t>(table) % 16 == 0) {
    const uint64_t wantv = (a.n / R + 255) / 256;
    const unsigned gridv = unsigned(std::max<uint64_t>(
        1, std::min<uint64_t>(wantv, uint64_t(di.sms) * 16)));
    if (offset_bytes == 4)
      launch_k(lm_eval_vec_kernel<int32_t>, gridv, 256, 0, st, a,
               static_cast<int32_t*>(table));
    else
      launch_k(lm_eval_vec_kernel<int64_t>, gridv, 256, 0, st, a,
               static_cast<int64_t*>(table));
    return check_launch();
  }
  if (offset_bytes == 4)
    launch_k(lm_eval_kernel<int32_t>, grid, 256, 0, st, a,
             static_cast<int32_t*>(table));
  else
    launch_k(lm_eval_kernel<int64_t>, grid, 256, 0, st, a,
             static_cast<int64_t*>(table));
  return check_launch();
}

}  // namespace lm

// ===========================================================================
// C ABI: device work
// ===========================================================================

extern "C" {

int lm_layout_copy(const lm_plan* plan, const void* src_dev,
                   int64_t src_capacity_elems, void* dst_dev,
                   int64_t dst_capacity_elems, void* cuda_stream) {
  try {
    if (!plan) return LM_E_INVALID;
    if (plan->size == 0) return LM_OK;
    if (!src_dev || !dst_dev) return LM_E_INVALID;
    if (src_capacity_elems < plan->src_cosize ||
        dst_capacity_elems < plan->dst_cosize)
      return LM_E_CAPACITY;
    const int64_t eb = plan->eb;
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(src_dev);
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(dst_dev);
    const uintptr_t s1 = s0 + uintptr_t(lm::mul_chk(plan->src_cosize, eb));
    const uintptr_t d1 = d0 + uintptr_t(lm::mul_chk(plan->dst_cosize, eb));
    if (s0 < d1 && d0 < s1) return LM_E_OVERLAP;
    const int64_t cap_bytes = lm::mul_chk(src_capacity_elems, eb);
    for (const lm::Piece& pc : plan->pieces) {
      const int rc = lm::launch_piece(*plan, pc, static_cast<const char*>(src_dev),
                                      cap_bytes, static_cast<char*>(dst_dev),
                                      cuda_stream);
      if (rc != LM_OK) return rc;
    }
    return LM_OK;
  } catch (const lm::Error& e) {
    return e.status;
  } catch (...) {
    return LM_E_INVALID;
  }
}

int lm_layout_copy_host(const lm_plan* plan, const void* src_host,
                        int64_t src_capacity_elems, void* dst_host,
                        int64_t dst_capacity_elems, void* src_dev,
                        void* dst_dev, void* cuda_stream) {
  try {
    if (!plan) return LM_E_INVALID;
    if (plan->size == 0) return LM_OK;
    if (!src_host || !dst_host || !src_dev || !dst_dev) return LM_E_INVALID;
    if (src_capacity_elems < plan->src_cosize ||
        dst_capacity_elems < plan->dst_cosize)
      return LM_E_CAPACITY;
    // a shard whose destination range holds other shards' elements cannot
    // download it without racing them
    if (!plan->dst_own) return LM_E_INVALID;
    const int64_t eb = plan->eb;
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    // a whole plan moves [0, capacity) up and [0, cosize) down; a shard
    // only the ranges its pieces reach
    const bool whole = plan->src_lo == 0 && plan->src_hi == plan->src_cosize;
    const int64_t in_lo = whole ? 0 : plan->src_lo;
    const int64_t in_hi = whole ? src_capacity_elems : plan->src_hi;
    const int64_t out_lo = plan->dst_lo, out_hi = plan->dst_hi;
    const size_t in_bytes = size_t(lm::mul_chk(in_hi - in_lo, eb));
    const size_t out_bytes = size_t(lm::mul_chk(out_hi - out_lo, eb));
    char* sd = static_cast<char*>(src_dev) + in_lo * eb;
    const char* sh = static_cast<const char*>(src_host) + in_lo * eb;
    char* dd = static_cast<char*>(dst_dev) + out_lo * eb;
    char* dh = static_cast<char*>(dst_host) + out_lo * eb;
    cudaError_t e = cudaSuccess;
    if (in_bytes)
      e = cudaMemcpyAsync(sd, sh, in_bytes, cudaMemcpyHostToDevice, st);
    // a destination with slots outside its image round-trips them
    if (e == cudaSuccess && out_bytes && plan->size < plan->dst_cosize)
      e = cudaMemcpyAsync(dd, dh, out_bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) {
      lm::set_cuda_error(int(e));
      return LM_E_CUDA;
    }
    const int rc = lm_layout_copy(plan, src_dev, src_capacity_elems, dst_dev,
                                  dst_capacity_elems, cuda_stream);
    if (rc != LM_OK) return rc;
    if (out_bytes)
      e = cudaMemcpyAsync(dh, dd, out_bytes, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) {
      lm::set_cuda_error(int(e));
      return LM_E_CUDA;
    }
    return LM_OK;
  } catch (const lm::Error& e) {
    return e.status;
  } catch (...) {
    return LM_E_INVALID;
  }
}

int lm_layout_eval_device(const lm_layout* layout, void* table_dev,
                          int offset_bytes, int64_t capacity,
                          void* cuda_stream) {
  try {
    if (!layout || (offset_bytes != 4 && offset_bytes != 8))
      return LM_E_INVALID;
    if (layout->size == 0) return LM_OK;
    if (!table_dev) return LM_E_INVALID;
    if (capacity < layout->size) return LM_E_CAPACITY;
    if (offset_bytes == 4 && layout->cosize - 1 > int64_t(0x7fffffff))
      return LM_E_OVERFLOW;
    return lm::launch_eval(*layout, table_dev, offset_bytes, cuda_stream);
  } catch (const lm::Error& e) {
    return e.status;
  } catch (...) {
    return LM_E_INVALID;
  }
}

int lm_last_cuda_error(void) { return lm::g_last_cuda; }

int lm_selftest_bounded_wait(int arrive, void* cuda_stream, int* status) {
  if (!status) return LM_E_INVALID;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  int before = 0;
  int rc = lm_device_status(cuda_stream, 1, &before);
  if (rc != LM_OK) return rc;
  lm::lm_selftest_wait_kernel<<<1, 32, 0, st>>>(arrive);
  rc = lm::check_launch();
  if (rc != LM_OK) return rc;
  return lm_device_status(cuda_stream, 1, status);
}

int lm_device_status(void* cuda_stream, int reset, int* status) {
  if (!status) return LM_E_INVALID;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  unsigned int word = 0;
  cudaError_t e = cudaStreamSynchronize(st);
  if (e == cudaSuccess)
    e = cudaMemcpyFromSymbol(&word, lm::g_lm_device_status, sizeof(word));
  if (e == cudaSuccess && reset && word) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(lm::g_lm_device_status, &zero, sizeof(zero));
  }
  if (e != cudaSuccess) {
    lm::set_cuda_error(int(e));
    return LM_E_CUDA;
  }
  *status = word ? LM_E_TIMEOUT : LM_OK;
  return LM_OK;
}

}  // extern "C"
