// The thread-value partitioned tile copy: grid-stride over tiles, load
// phase into a shared tile, store phase out of it, both through the device
// functions of layoutmove_tv.cuh -- the building block this kernel exists
// to run and test.  With two shared tiles (`two`), the loads of a block's
// next tile are in flight while it stores the current one.

#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

#include <cstdlib>

#include "layoutmove_tv.cuh"
#include "lm_internal.h"
#include "lm_mbar.cuh"

namespace lm {
namespace {

template <int VL, int VS>
__global__ void __launch_bounds__(1024)
    lm_tv_kernel(const __grid_constant__ lm_tv_args a,
                 const char* __restrict__ src, char* __restrict__ dst,
                 int two) {
  extern __shared__ __align__(16) char tile_smem[];
  const int t = int(threadIdx.x);
  const int64_t step = gridDim.x;
  int64_t tile = blockIdx.x;
  if (tile >= a.n_tiles) return;  // whole block
  const lm_tv::Bases b = lm_tv::thread_bases(a, t);
  int64_t sb, db;
  lm_tv::tile_bases(a, tile, &sb, &db);
  if (two) {
    lm_tv::load_tile<VL>(a, b, src, tile_smem, sb, t);
    lm_tv::commit_copies();
  }
  for (int i = 0; tile < a.n_tiles; ++i, tile += step) {
    char* cur = tile_smem + (two ? (i & 1) * a.smem_bytes : 0);
    const int64_t next = tile + step;
    int64_t nsb = 0, ndb = 0;
    if (next < a.n_tiles) lm_tv::tile_bases(a, next, &nsb, &ndb);
    if (two) {
      // the other tile was last read before the barrier that ended the
      // previous iteration
      if (next < a.n_tiles)
        lm_tv::load_tile<VL>(a, b, src,
                             tile_smem + ((i + 1) & 1) * a.smem_bytes, nsb, t);
      lm_tv::commit_copies();
      lm_tv::wait_copies_but<1>();  // this tile's group has landed
    } else {
      lm_tv::load_tile<VL>(a, b, src, cur, sb, t);
      lm_tv::wait_copies();
    }
    __syncthreads();
    lm_tv::store_tile<VS>(a, b, cur, dst, db, t);
    __syncthreads();
    sb = nsb;
    db = ndb;
  }
}

// The same loop with every tile-invariant offset in registers (phases of
// at most MAXV values per thread, in-tile offsets within 31 bits, blocks
// of at most 512 threads), with NS shared tiles: the loads of a block's
// next NS-1 tiles are in flight while it stores the current one.  Every
// iteration commits one group of copies (possibly empty), so waiting until
// at most NS-1 groups are pending means the current tile has landed.
template <int VL, int VS, int MAXV, int NS>
__global__ void __launch_bounds__(512)
    lm_tv_cached_kernel(const __grid_constant__ lm_tv_args a,
                        const char* __restrict__ src, char* __restrict__ dst,
                        int /*unused*/) {
  extern __shared__ __align__(16) char tile_smem[];
  const int t = int(threadIdx.x);
  const int64_t stride = gridDim.x;
  const int64_t first = blockIdx.x;
  if (first >= a.n_tiles) return;  // whole block
  lm_tv::Offsets<MAXV> o;
  lm_tv::thread_offsets<MAXV>(a, lm_tv::thread_bases(a, t), o);
  int64_t sb, db;
#pragma unroll
  for (int k = 0; k < NS - 1; ++k) {
    const int64_t tile = first + k * stride;
    if (tile < a.n_tiles) {
      lm_tv::tile_bases(a, tile, &sb, &db);
      lm_tv::load_tile<VL, MAXV>(a, o, src, tile_smem + k * a.smem_bytes, sb,
                                 t);
    }
    lm_tv::commit_copies();
  }
  int slot = 0;  // the shared tile of the current tile
  for (int64_t tile = first; tile < a.n_tiles; tile += stride) {
    const int64_t ahead = tile + (NS - 1) * stride;
    // the ahead slot was last read before the barrier ending the previous
    // iteration
    const int aslot = slot == 0 ? NS - 1 : slot - 1;
    if (ahead < a.n_tiles) {
      lm_tv::tile_bases(a, ahead, &sb, &db);
      lm_tv::load_tile<VL, MAXV>(a, o, src, tile_smem + aslot * a.smem_bytes,
                                 sb, t);
    }
    lm_tv::commit_copies();
    lm_tv::wait_copies_but<NS - 1>();
    __syncthreads();
    lm_tv::tile_bases(a, tile, &sb, &db);
    lm_tv::store_tile<VS, MAXV>(a, o, tile_smem + slot * a.smem_bytes, dst,
                                db, t);
    __syncthreads();
    slot = slot + 1 == NS ? 0 : slot + 1;
  }
}

// The cached loop without block-wide barriers: NS shared tiles, each with
// a "full" mbarrier that every loading thread's cp.async copies of the
// tile arrive on when they land (cp.async.mbarrier.arrive.noinc) and an
// "empty" mbarrier every storing thread arrives on once it has read the
// tile.  A thread loads tile i + NS - 1 after the storers released its
// stage, then waits for tile i to be full and stores its share; warps run
// ahead of each other up to the pipeline depth.  Every wait is bounded: a
// thread that gives up records it in the device status word, waits for its
// own copies (a hardware wait) and leaves.  Load phases of 4-, 8- and
// 16-byte vectors only (all of them cp.async).
template <int VL, int VS, int MAXV, int NS>
__global__ void __launch_bounds__(512)
    lm_tv_mbar_kernel(const __grid_constant__ lm_tv_args a,
                      const char* __restrict__ src, char* __restrict__ dst,
                      unsigned int* status) {
  extern __shared__ __align__(128) char smem_raw[];
  const uint32_t bars = uint32_t(__cvta_generic_to_shared(smem_raw));
  auto full = [&](int s) { return bars + 8u * uint32_t(s); };
  auto empty = [&](int s) { return bars + 8u * uint32_t(NS + s); };
  char* tiles = smem_raw + 128;
  const int t = int(threadIdx.x);
  const bool loader = t < a.load.n_thr, storer = t < a.store.n_thr;
  if (t == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      mbar_init(full(s), uint32_t(a.load.n_thr));
      mbar_init(empty(s), uint32_t(a.store.n_thr));
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  const int64_t first = blockIdx.x, stride = gridDim.x;
  if (first >= a.n_tiles) return;  // whole block
  const int64_t n_local = (a.n_tiles - first + stride - 1) / stride;
  lm_tv::Offsets<MAXV> o;
  lm_tv::thread_offsets<MAXV>(a, lm_tv::thread_bases(a, t), o);
  bool ok = true;
  // tile number i of this block into stage i % NS
  auto issue = [&](int64_t i) -> bool {
    const int s = int(i % NS);
    if (i >= NS && !mbar_wait(empty(s), uint32_t((i / NS) - 1) & 1u))
      return false;
    int64_t sb, db;
    lm_tv::tile_bases(a, first + i * stride, &sb, &db);
    lm_tv::load_tile<VL, MAXV>(a, o, src, tiles + s * a.smem_bytes, sb, t);
    cp_async_arrive_noinc(full(s));
    return true;
  };
  if (loader)
    for (int64_t i = 0; i < NS - 1 && i < n_local && ok; ++i) ok = issue(i);
  for (int64_t i = 0; i < n_local && ok; ++i) {
    if (loader && i + NS - 1 < n_local) ok = issue(i + NS - 1);
    if (!ok) break;
    if (storer) {
      const int s = int(i % NS);
      if (!mbar_wait(full(s), uint32_t(i / NS) & 1u)) {
        ok = false;
        break;
      }
      int64_t sb, db;
      lm_tv::tile_bases(a, first + i * stride, &sb, &db);
      lm_tv::store_tile<VS, MAXV>(a, o, tiles + s * a.smem_bytes, dst, db, t);
      mbar_arrive(empty(s));
    }
  }
  if (!ok && status) atomicOr(status, 1u);
  lm_tv::wait_copies();  // no copy of this thread outlives it
}

typedef void (*TvKernel)(const lm_tv_args, const char*, char*, int);
typedef void (*TvMbarKernel)(const lm_tv_args, const char*, char*,
                             unsigned int*);

template <int VL, int NS>
TvMbarKernel pick_mbar_store(int vs) {
  switch (vs) {
    case 4: return lm_tv_mbar_kernel<VL, 4, 4, NS>;
    case 8: return lm_tv_mbar_kernel<VL, 8, 4, NS>;
    case 16: return lm_tv_mbar_kernel<VL, 16, 4, NS>;
  }
  return nullptr;
}

template <int NS>
TvMbarKernel pick_mbar_ns(int vl, int vs) {
  switch (vl) {
    case 4: return pick_mbar_store<4, NS>(vs);
    case 8: return pick_mbar_store<8, NS>(vs);
    case 16: return pick_mbar_store<16, NS>(vs);
  }
  return nullptr;
}

// The mbarrier pipeline (LM_TV_MBAR=1; the barrier-paced kernels by
// default) and its depth (LM_TV_STAGES, 2..4).  Measured on GB300 it ran
// the bench's tile copies as fast as the barrier-paced kernels, no faster
// (54.8 against 53.6 us for the 8192^2 bf16 tiling, 29.0 against 29.1 us for
// the fp32 transpose with 16-byte loads), at any depth.
int tv_mbar_stages() {
  static const int v = [] {
    const char* e = std::getenv("LM_TV_MBAR");
    if (!e || e[0] != '1') return 0;
    const char* d = std::getenv("LM_TV_STAGES");
    const int n = d ? std::atoi(d) : 3;
    return n < 2 ? 2 : (n > 4 ? 4 : n);
  }();
  return v;
}

TvMbarKernel pick_mbar(int vl, int vs, int ns) {
  switch (ns) {
    case 2: return pick_mbar_ns<2>(vl, vs);
    case 4: return pick_mbar_ns<4>(vl, vs);
    default: return pick_mbar_ns<3>(vl, vs);
  }
}

template <int VL>
TvKernel pick_cached_store(int vs) {
  switch (vs) {
    case 4: return lm_tv_cached_kernel<VL, 4, 4, 2>;
    case 8: return lm_tv_cached_kernel<VL, 8, 4, 2>;
    case 16: return lm_tv_cached_kernel<VL, 16, 4, 2>;
  }
  return nullptr;
}

// Two shared tiles per block: three and four measured 4% and 8% slower on
// the 8192^2 bf16 tiling, and so did moving two tiles between barriers.
TvKernel pick_cached(int vl, int vs) {
  switch (vl) {
    case 4: return pick_cached_store<4>(vs);
    case 8: return pick_cached_store<8>(vs);
    case 16: return pick_cached_store<16>(vs);
  }
  return nullptr;
}

template <int VL>
TvKernel pick_store(int vs) {
  switch (vs) {
    case 1: return lm_tv_kernel<VL, 1>;
    case 2: return lm_tv_kernel<VL, 2>;
    case 4: return lm_tv_kernel<VL, 4>;
    case 8: return lm_tv_kernel<VL, 8>;
    case 16: return lm_tv_kernel<VL, 16>;
  }
  return nullptr;
}

TvKernel pick(int vl, int vs) {
  switch (vl) {
    case 1: return pick_store<1>(vs);
    case 2: return pick_store<2>(vs);
    case 4: return pick_store<4>(vs);
    case 8: return pick_store<8>(vs);
    case 16: return pick_store<16>(vs);
  }
  return nullptr;
}

int fail_cuda(cudaError_t e) {
  set_cuda_error(int(e));
  return LM_E_CUDA;
}

// Dynamic shared memory above 48 KiB needs an opt-in per device and kernel.
cudaError_t allow_tv_smem(const void* k, int dev, int smem) {
  if (smem <= 49152) return cudaSuccess;
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, int> done;
  std::lock_guard<std::mutex> g(mu);
  const auto key = std::make_pair(dev, k);
  auto it = done.find(key);
  if (it == done.end() || it->second < smem) {
    const cudaError_t e = cudaFuncSetAttribute(
        k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    done[key] = smem;
  }
  return cudaSuccess;
}

// Blocks per resident slot (LM_TV_WAVES, default 1: one persistent wave
// that strides over the tiles).
int64_t tv_waves() {
  static const int64_t v = [] {
    const char* e = std::getenv("LM_TV_WAVES");
    const long long w = e ? std::atoll(e) : 1;
    return int64_t(w < 1 ? 1 : w);
  }();
  return v;
}

// One block per resident slot at most, grid-stride over the tiles.
int launch_mbar(TvMbarKernel k, const lm_tv_args& a, const char* src,
                char* dst, void* stream, int smem, unsigned int* status) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  e = allow_tv_smem(reinterpret_cast<const void*>(k), dev, smem);
  if (e != cudaSuccess) return fail_cuda(e);
  int sms = 0, per_sm = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail_cuda(e);
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k,
                                                    a.block_threads,
                                                    size_t(smem));
  if (e != cudaSuccess) return fail_cuda(e);
  if (per_sm < 1) return LM_E_INVALID;  // the block cannot be resident
  const int64_t resident = int64_t(sms) * per_sm * tv_waves();
  const unsigned grid =
      unsigned(a.n_tiles < resident ? a.n_tiles : resident);
  k<<<grid, unsigned(a.block_threads), size_t(smem),
      static_cast<cudaStream_t>(stream)>>>(a, src, dst, status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e);
  return LM_OK;
}

}  // namespace

int launch_tv(const lm_tv_plan& plan, const char* src, char* dst,
              void* stream) {
  const lm_tv_args& a = plan.args;
  if (a.n_tiles == 0) return LM_OK;
  const int most = a.load.n_val > a.store.n_val ? a.load.n_val : a.store.n_val;
  const int ns = tv_mbar_stages();
  if (ns && a.offsets32 && a.block_threads <= 512 && most <= 4 &&
      128 + ns * int64_t(a.smem_bytes) <= 232448 && a.smem_bytes % 16 == 0) {
    const TvMbarKernel mk =
        pick_mbar(a.load.vec_bytes, a.store.vec_bytes, ns);
    unsigned int* status = device_status_word();
    if (mk && status)
      return launch_mbar(mk, a, src, dst, stream, 128 + ns * a.smem_bytes,
                         status);
  }
  TvKernel k = nullptr;
  int smem = 0, two = 0;
  if (a.offsets32 && a.block_threads <= 512 && most <= 4 &&
      2 * int64_t(a.smem_bytes) <= 232448) {
    k = pick_cached(a.load.vec_bytes, a.store.vec_bytes);
    smem = 2 * a.smem_bytes;
  }
  if (!k) {
    k = pick(a.load.vec_bytes, a.store.vec_bytes);
    // two shared tiles when they fit beside each other
    two = 2 * int64_t(a.smem_bytes) <= 232448 && a.n_tiles > 1 ? 1 : 0;
    smem = a.smem_bytes * (two ? 2 : 1);
  }
  if (!k) return LM_E_INVALID;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (smem > 49152) {
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, int> done;
    std::lock_guard<std::mutex> g(mu);
    const auto key = std::make_pair(dev, reinterpret_cast<const void*>(k));
    auto it = done.find(key);
    if (it == done.end() || it->second < smem) {
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               smem);
      if (e != cudaSuccess) return fail_cuda(e);
      done[key] = smem;
    }
  }
  int sms = 0, per_sm = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail_cuda(e);
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k,
                                                    a.block_threads,
                                                    size_t(smem));
  if (e != cudaSuccess) return fail_cuda(e);
  if (per_sm < 1) return LM_E_INVALID;  // the block cannot be resident
  const int64_t resident = int64_t(sms) * per_sm * tv_waves();
  const unsigned grid =
      unsigned(a.n_tiles < resident ? a.n_tiles : resident);
  k<<<grid, unsigned(a.block_threads), size_t(smem),
      static_cast<cudaStream_t>(stream)>>>(a, src, dst, two);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e);
  return LM_OK;
}

}  // namespace lm

extern "C" int lm_tv_copy(const lm_tv_plan* plan, const void* src_dev,
                          int64_t src_capacity_elems, void* dst_dev,
                          int64_t dst_capacity_elems, void* cuda_stream) {
  try {
    if (!plan) return LM_E_INVALID;
    const lm_tv_args& a = plan->args;
    if (a.n_tiles == 0) return LM_OK;
    if (!src_dev || !dst_dev) return LM_E_INVALID;
    if (src_capacity_elems < plan->src_cosize ||
        dst_capacity_elems < plan->dst_cosize)
      return LM_E_CAPACITY;
    const int64_t eb = a.elem_bytes;
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(src_dev);
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(dst_dev);
    if (s0 % uintptr_t(a.load.vec_bytes) || d0 % uintptr_t(a.store.vec_bytes) ||
        s0 % uintptr_t(eb) || d0 % uintptr_t(eb))
      return LM_E_INVALID;
    const uintptr_t s1 = s0 + uintptr_t(lm::mul_chk(plan->src_cosize, eb));
    const uintptr_t d1 = d0 + uintptr_t(lm::mul_chk(plan->dst_cosize, eb));
    if (s0 < d1 && d0 < s1) return LM_E_OVERLAP;
    return lm::launch_tv(*plan, static_cast<const char*>(src_dev),
                         static_cast<char*>(dst_dev), cuda_stream);
  } catch (const lm::Error& e) {
    return e.status;
  } catch (...) {
    return LM_E_INVALID;
  }
}
