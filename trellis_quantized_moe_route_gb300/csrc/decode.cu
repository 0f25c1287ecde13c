// Stand-alone trellis tile decode into memory, for bit-exact parity checks of
// the decoder the GEMM kernels use (the product path never materialises
// weights). One thread per run of 8 states; output in weight order j.
#include "launch.h"

namespace tmoe {

template <int K>
__device__ __forceinline__ void decode_run(const uint16_t* tile, int run, uint32_t (&s)[8]) {
  const int row = run >> 1, h = run & 1;
  if (K == 4) {
    uint32_t p, c;
    run_load_k4(tile, row, h, p, c);
    run_states_k4(p, c, s);
  } else {
    uint32_t hi, lo;
    int off;
    run_window_generic<K>(tile, 8 * run, hi, lo, off);
    run_states_generic<K>(hi, lo, off, s);
  }
}

template <int K, bool E4M3>
__global__ void __launch_bounds__(256) k_decode_tiles(const uint16_t* __restrict__ tiles, int ntiles, void* __restrict__ dst) {
  const long gid = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (long)ntiles * 32) return;
  const long t = gid >> 5;
  const int run = (int)(gid & 31);
  uint32_t s[8];
  decode_run<K>(tiles + t * 16 * K, run, s);
  if (!E4M3) {
    uint32_t w[4];
    run_weights_f16(s, w);
    uint4 o = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(dst) + t * 256 + run * 8)[0] = o;
  } else {
    uint32_t qv[2];
    run_weights_e4m3(s, qv);
    reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(dst) + t * 256 + run * 8)[0] = make_uint2(qv[0], qv[1]);
  }
}

template <int K>
static cudaError_t launch_k(const int16_t* tiles, int ntiles, bool e4m3, void* dst, cudaStream_t st) {
  const long threads = (long)ntiles * 32;
  const int blocks = (int)((threads + 255) / 256);
  const uint16_t* t = reinterpret_cast<const uint16_t*>(tiles);
  if (e4m3)
    k_decode_tiles<K, true><<<blocks, 256, 0, st>>>(t, ntiles, dst);
  else
    k_decode_tiles<K, false><<<blocks, 256, 0, st>>>(t, ntiles, dst);
  return cudaGetLastError();
}

cudaError_t launch_decode_tiles(const int16_t* tiles, int K, int ntiles, bool e4m3, void* dst, cudaStream_t st) {
  if (ntiles == 0) return cudaSuccess;
  switch (K) {
    case 2: return launch_k<2>(tiles, ntiles, e4m3, dst, st);
    case 3: return launch_k<3>(tiles, ntiles, e4m3, dst, st);
    case 4: return launch_k<4>(tiles, ntiles, e4m3, dst, st);
    case 5: return launch_k<5>(tiles, ntiles, e4m3, dst, st);
    case 6: return launch_k<6>(tiles, ntiles, e4m3, dst, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tmoe
