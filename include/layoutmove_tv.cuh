// layoutmove_tv.cuh -- device side of the thread-value partitioned tile
// copy (layoutmove_tv.h describes the arguments).
//
// A building block for kernels that stage tiles through shared memory: with
// the lm_tv_args a plan produced (lm_tv_plan_args), a block
//
//     lm_tv::load_tile<VL>(a, src, smem, src_tile_base, threadIdx.x);
//     lm_tv::wait_copies();
//     __syncthreads();
//     ... use the shared tile ...
//     lm_tv::store_tile<VS>(a, smem, dst, dst_tile_base, threadIdx.x);
//
// where VL / VS are a.load.vec_bytes / a.store.vec_bytes and the tile bases
// come from lm_tv::tile_bases.  Thread t moves its local_partition of the
// grouped tile ("CUTLASS Layout可视化" §5.3): value v of the load phase goes
// from src[Swz_src(src_tile_base + base_from(t) + from_val[v])] to
// smem[Swz_smem(base_to(t) + to_val[v])], in elements.  4-, 8- and 16-byte
// loads use cp.async (asynchronous: wait_copies() before the tile is read);
// narrower ones plain loads and stores.  `src` and `dst` must be aligned to
// the phase's vector bytes, `smem` to 16 bytes.
//
// Pass the arguments as `const __grid_constant__ lm_tv_args` so the value
// tables are read from the parameter bank rather than copied per thread.
#ifndef LAYOUTMOVE_TV_CUH
#define LAYOUTMOVE_TV_CUH

#include <stdint.h>

#include "layoutmove_tv.h"

namespace lm_tv {

// Swizzle<B,M,S> on an element offset ("CUTLASS Layout可视化" §4.3).
__device__ __forceinline__ int64_t swizzle(int64_t o, const int32_t* z) {
  if (z[0] == 0) return o;
  const int64_t mask = ((int64_t(1) << z[0]) - 1) << z[1];
  return o ^ ((o >> z[2]) & mask);
}

// Element offsets of tile `tile` (colex over the grid modes) in src and dst.
__device__ __forceinline__ void tile_bases(const lm_tv_args& a, int64_t tile,
                                           int64_t* src_base,
                                           int64_t* dst_base) {
  int64_t s = 0, d = 0;
  for (int k = 0; k < a.n_grid; ++k) {
    const int64_t c = tile % a.grid_ext[k];
    tile /= a.grid_ext[k];
    s += c * a.grid_src[k];
    d += c * a.grid_dst[k];
  }
  *src_base = s;
  *dst_base = d;
}

// base_from(t), base_to(t) of one phase.
__device__ __forceinline__ void thread_bases(const lm_tv_phase& p, int t,
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

// Load phase: this thread's values of the tile at src_tile_base.
template <int VB>
__device__ __forceinline__ void load_tile(const lm_tv_args& a,
                                          const char* src, char* smem,
                                          int64_t src_tile_base, int t) {
  const lm_tv_phase& p = a.load;
  if (t >= p.n_thr) return;
  int32_t bf, bt;
  thread_bases(p, t, &bf, &bt);
  const int64_t eb = a.elem_bytes;
  const int64_t gbase = src_tile_base + bf;
#pragma unroll 4
  for (int v = 0; v < p.n_val; ++v) {
    const int64_t go = swizzle(gbase + p.from_val[v], a.src_swz);
    const int64_t so = swizzle(int64_t(bt) + p.to_val[v], a.smem_swz);
    copy_to_shared<VB>(smem + so * eb, src + go * eb);
  }
}

// Store phase: this thread's values of the shared tile to the tile at
// dst_tile_base.
template <int VB>
__device__ __forceinline__ void store_tile(const lm_tv_args& a,
                                           const char* smem, char* dst,
                                           int64_t dst_tile_base, int t) {
  typedef typename Word<VB>::T T;
  const lm_tv_phase& p = a.store;
  if (t >= p.n_thr) return;
  int32_t bf, bt;
  thread_bases(p, t, &bf, &bt);
  const int64_t eb = a.elem_bytes;
  const int64_t gbase = dst_tile_base + bt;
#pragma unroll 4
  for (int v = 0; v < p.n_val; ++v) {
    const int64_t so = swizzle(int64_t(bf) + p.from_val[v], a.smem_swz);
    const int64_t go = swizzle(gbase + p.to_val[v], a.dst_swz);
    *reinterpret_cast<T*>(dst + go * eb) =
        *reinterpret_cast<const T*>(smem + so * eb);
  }
}

}  // namespace lm_tv

#endif  // LAYOUTMOVE_TV_CUH
