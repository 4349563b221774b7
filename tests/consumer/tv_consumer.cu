// A consumer kernel compiled apart from the library: it stages tiles with
// the device functions of include/layoutmove_tv.cuh, complements every byte
// of the shared tile, and stores the tile with the same functions.  Used by
// tests/test_gpu_tv.py to show the building block works in kernels of
// their own.
#include <cuda_runtime.h>

#include <cstring>

#include "layoutmove_tv.cuh"

__global__ void tv_consumer_kernel(const __grid_constant__ lm_tv_args a,
                                   const char* __restrict__ src,
                                   char* __restrict__ dst) {
  extern __shared__ __align__(16) char sm[];
  const int t = int(threadIdx.x);
  const lm_tv::Bases b = lm_tv::thread_bases(a, t);
  for (int64_t tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x) {
    int64_t sb, db;
    lm_tv::tile_bases(a, tile, &sb, &db);
    lm_tv::load_tile<16>(a, b, src, sm, sb, t);
    lm_tv::wait_copies();
    __syncthreads();
    for (int i = t; i < a.smem_bytes; i += int(blockDim.x))
      sm[i] = char(~sm[i]);
    __syncthreads();
    lm_tv::store_tile<16>(a, b, sm, dst, db, t);
    __syncthreads();
  }
}

extern "C" int tv_consumer_launch(const void* args, const void* src,
                                  void* dst, int blocks, void* stream) {
  lm_tv_args a;
  std::memcpy(&a, args, sizeof(a));
  if (a.load.vec_bytes != 16 || a.store.vec_bytes != 16 || blocks < 1)
    return -1;
  if (a.smem_bytes > 49152) return -1;
  tv_consumer_kernel<<<blocks, a.block_threads, size_t(a.smem_bytes),
                       static_cast<cudaStream_t>(stream)>>>(
      a, static_cast<const char*>(src), static_cast<char*>(dst));
  return int(cudaGetLastError());
}
