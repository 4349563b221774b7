// layoutmove_tv.cuh -- device side of the thread-value partitioned tile
// copy (layoutmove_tv.h describes the arguments).
//
// A building block for kernels that stage tiles through shared memory: with
// the lm_tv_args a plan produced (lm_tv_plan_args), a block
//
//     const lm_tv::Bases b = lm_tv::thread_bases(a, threadIdx.x);  // once
//     for (each tile) {
//       lm_tv::tile_bases(a, tile, &src_base, &dst_base);
//       lm_tv::load_tile<VL>(a, b, src, smem, src_base, threadIdx.x);
//       lm_tv::wait_copies();
//       __syncthreads();
//       ... use the shared tile ...
//       lm_tv::store_tile<VS>(a, b, smem, dst, dst_base, threadIdx.x);
//       __syncthreads();
//     }
//
// where VL / VS are a.load.vec_bytes / a.store.vec_bytes.  When both phases
// have at most MAXV values per thread and a.offsets32 is set, the overloads
// taking an Offsets<MAXV> (filled once by thread_offsets) keep every
// tile-invariant offset in registers instead.  Thread t moves
// its local_partition of the grouped tile ("CUTLASS Layout可视化" §5.3):
// value v of the load phase goes from src + Swz_src(src_base + base_from(t)
// + from_val[v]) to smem + Swz_smem(base_to(t) + to_val[v]), all in bytes.
// 4-, 8- and 16-byte loads use cp.async (asynchronous: wait_copies() before
// the tile is read, or commit_copies() / wait_copies_but<N>() to keep later
// tiles' loads in flight); narrower ones plain loads and stores.  `src` and `dst`
// must be aligned to the phase's vector bytes, `smem` to 16 bytes.
//
// Pass the arguments as `const __grid_constant__ lm_tv_args` so the value
// tables are read from the parameter bank rather than copied per thread.
// Needs C++17 (nvcc -std=c++17) and cp.async (sm_80 or later; the library
// builds it for sm_103a).
#ifndef LAYOUTMOVE_TV_CUH
#define LAYOUTMOVE_TV_CUH

#include <stdint.h>

#include "layoutmove_tv.h"

namespace lm_tv {

// Swizzle<B,M,S> on a byte offset ("CUTLASS Layout可视化" §4.3).
__device__ __forceinline__ int64_t swizzle(int64_t o, const int32_t* z) {
  if (z[0] == 0) return o;
  const int64_t mask = ((int64_t(1) << z[0]) - 1) << z[1];
  return o ^ ((o >> z[2]) & mask);
}

__device__ __forceinline__ uint32_t fast_div(uint32_t n,
                                             const lm_tv_fastdiv& f) {
  const uint32_t t = __umulhi(f.m, n);
  return (t + ((n - t) >> f.s1)) >> f.s2;
}

// Byte offsets of tile `tile` (colex over the grid modes) in src and dst.
__device__ __forceinline__ void tile_bases(const lm_tv_args& a, int64_t tile,
                                           int64_t* src_base,
                                           int64_t* dst_base) {
  int64_t s = 0, d = 0;
  if (a.grid_fast) {
    uint32_t rem = uint32_t(tile);
    for (int k = 0; k < a.n_grid; ++k) {
      const uint32_t q = fast_div(rem, a.grid_div[k]);
      const uint32_t c = rem - q * a.grid_div[k].d;
      rem = q;
      s += int64_t(c) * a.grid_src[k];
      d += int64_t(c) * a.grid_dst[k];
    }
  } else {
    for (int k = 0; k < a.n_grid; ++k) {
      const int64_t c = tile % a.grid_ext[k];
      tile /= a.grid_ext[k];
      s += c * a.grid_src[k];
      d += c * a.grid_dst[k];
    }
  }
  *src_base = s;
  *dst_base = d;
}

// A thread's base offsets in both phases (computed once per thread).
struct Bases {
  int32_t load_from, load_to, store_from, store_to;
};

__device__ __forceinline__ void phase_bases(const lm_tv_phase& p, int t,
                                            int32_t* from, int32_t* to) {
  int32_t f = 0, g = 0;
  for (int j = 0; j < p.n_leaves; ++j) {
    const int32_t c = (t / p.leaf_stride[j]) % p.leaf_ext[j];
    f += c * p.from_step[j];
    g += c * p.to_step[j];
  }
  *from = f;
  *to = g;
}

__device__ __forceinline__ Bases thread_bases(const lm_tv_args& a, int t) {
  Bases b;
  phase_bases(a.load, t, &b.load_from, &b.load_to);
  phase_bases(a.store, t, &b.store_from, &b.store_to);
  return b;
}

// Swizzle of an offset inside the shared tile (32-bit).
__device__ __forceinline__ int32_t swizzle32(int32_t o, const int32_t* z) {
  if (z[0] == 0) return o;
  return o ^ ((o >> z[2]) & (((1 << z[0]) - 1) << z[1]));
}

template <int VB> struct Word;
template <> struct Word<1> { typedef uint8_t T; };
template <> struct Word<2> { typedef uint16_t T; };
template <> struct Word<4> { typedef uint32_t T; };
template <> struct Word<8> { typedef uint2 T; };
template <> struct Word<16> { typedef uint4 T; };

template <int VB>
__device__ __forceinline__ void copy_to_shared(char* smem, const char* g) {
  if constexpr (VB >= 4) {
    const uint32_t s = uint32_t(__cvta_generic_to_shared(smem));
    if constexpr (VB == 16)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s),
                   "l"(g)
                   : "memory");
    else
      asm volatile("cp.async.ca.shared.global [%0], [%1], %2;\n" ::"r"(s),
                   "l"(g), "n"(VB)
                   : "memory");
  } else {
    typedef typename Word<VB>::T T;
    *reinterpret_cast<T*>(smem) = *reinterpret_cast<const T*>(g);
  }
}

__device__ __forceinline__ void wait_copies() {
  asm volatile("cp.async.wait_all;\n" ::: "memory");
}

// Pipelining: close the group of copies issued so far, and wait until at
// most N of the closed groups are still in flight.
__device__ __forceinline__ void commit_copies() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void wait_copies_but() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Load phase: this thread's values of the tile at src_tile_base.
template <int VB>
__device__ __forceinline__ void load_tile(const lm_tv_args& a, const Bases& b,
                                          const char* src, char* smem,
                                          int64_t src_tile_base, int t) {
  const lm_tv_phase& p = a.load;
  if (t >= p.n_thr) return;
  const int64_t gbase = src_tile_base + b.load_from;
#pragma unroll 4
  for (int v = 0; v < p.n_val; ++v) {
    const int64_t go = swizzle(gbase + p.from_val[v], a.src_swz);
    const int32_t so = swizzle32(b.load_to + p.to_val[v], a.smem_swz);
    copy_to_shared<VB>(smem + so, src + go);
  }
}

// Store phase: this thread's values of the shared tile to the tile at
// dst_tile_base.
template <int VB>
__device__ __forceinline__ void store_tile(const lm_tv_args& a, const Bases& b,
                                           const char* smem, char* dst,
                                           int64_t dst_tile_base, int t) {
  typedef typename Word<VB>::T T;
  const lm_tv_phase& p = a.store;
  if (t >= p.n_thr) return;
  const int64_t gbase = dst_tile_base + b.store_to;
#pragma unroll 4
  for (int v = 0; v < p.n_val; ++v) {
    const int32_t so = swizzle32(b.store_from + p.from_val[v], a.smem_swz);
    const int64_t go = swizzle(gbase + p.to_val[v], a.dst_swz);
    *reinterpret_cast<T*>(dst + go) = *reinterpret_cast<const T*>(smem + so);
  }
}

// ---------------------------------------------------------------------------
// The same phases with every tile-invariant offset computed once per thread
// (for phases of at most MAXV values per thread): the shared offsets
// swizzled, and the global in-tile offsets swizzled when the side's swizzle
// commutes with the tile base.  Per value a tile then costs one add.
// ---------------------------------------------------------------------------

template <int MAXV>
struct Offsets {
  int32_t load_g[MAXV], load_s[MAXV];    // global (in-tile), shared
  int32_t store_s[MAXV], store_g[MAXV];  // shared, global (in-tile)
};

template <int MAXV>
__device__ __forceinline__ void thread_offsets(const lm_tv_args& a,
                                               const Bases& b,
                                               Offsets<MAXV>& o) {
#pragma unroll
  for (int v = 0; v < MAXV; ++v) {
    o.load_g[v] = o.load_s[v] = o.store_s[v] = o.store_g[v] = 0;
    if (v < a.load.n_val) {
      const int64_t g = int64_t(b.load_from) + a.load.from_val[v];
      o.load_g[v] = int32_t(a.src_swz_tile ? swizzle(g, a.src_swz) : g);
      o.load_s[v] = swizzle32(b.load_to + a.load.to_val[v], a.smem_swz);
    }
    if (v < a.store.n_val) {
      o.store_s[v] = swizzle32(b.store_from + a.store.from_val[v], a.smem_swz);
      const int64_t g = int64_t(b.store_to) + a.store.to_val[v];
      o.store_g[v] = int32_t(a.dst_swz_tile ? swizzle(g, a.dst_swz) : g);
    }
  }
}

template <int VB, int MAXV>
__device__ __forceinline__ void load_tile(const lm_tv_args& a,
                                          const Offsets<MAXV>& o,
                                          const char* src, char* smem,
                                          int64_t src_tile_base, int t) {
  if (t >= a.load.n_thr) return;
#pragma unroll
  for (int v = 0; v < MAXV; ++v) {
    if (v >= a.load.n_val) break;
    int64_t go = src_tile_base + o.load_g[v];
    if (!a.src_swz_tile) go = swizzle(go, a.src_swz);
    copy_to_shared<VB>(smem + o.load_s[v], src + go);
  }
}

template <int VB, int MAXV>
__device__ __forceinline__ void store_tile(const lm_tv_args& a,
                                           const Offsets<MAXV>& o,
                                           const char* smem, char* dst,
                                           int64_t dst_tile_base, int t) {
  typedef typename Word<VB>::T T;
  if (t >= a.store.n_thr) return;
#pragma unroll
  for (int v = 0; v < MAXV; ++v) {
    if (v >= a.store.n_val) break;
    int64_t go = dst_tile_base + o.store_g[v];
    if (!a.dst_swz_tile) go = swizzle(go, a.dst_swz);
    *reinterpret_cast<T*>(dst + go) =
        *reinterpret_cast<const T*>(smem + o.store_s[v]);
  }
}

}  // namespace lm_tv

#endif  // LAYOUTMOVE_TV_CUH
