// Weight-only quantized matrices formed as fp16 (for the prefill phases,
// whose tcgen05 GEMMs take fp16 operands from shared memory):
//   INT8  w[o][i] = fp16(scale[o] * q[o][i])
//   int4  w[o][i] = fp16(scale[o][i / g] * (c(o, i) - zero[o][i / g]))
// The code arithmetic is exact in fp32 (a code has at most 8 bits, a scale
// 11), so the result is the product rounded once to fp16, the same value
// the decode kernel forms in registers.
#include "common.cuh"
#include "kernels.h"

namespace blk {
namespace {

__global__ void dequant_i8_kernel(const int8_t* q, const __half* scale, int64_t rows, int64_t K,
                                  __half* w) {
  const int64_t n4 = rows * K / 4;   // K % 16 == 0
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const char4 c = reinterpret_cast<const char4*>(q)[i];
    const float s = __half2float(scale[(4 * i) / K]);
    __half2* o = reinterpret_cast<__half2*>(w) + 2 * i;
    o[0] = __floats2half2_rn(s * (float)c.x, s * (float)c.y);
    o[1] = __floats2half2_rn(s * (float)c.z, s * (float)c.w);
  }
}

__global__ void dequant_u4_kernel(const uint8_t* packed, const __half* scale,
                                  const uint8_t* zero, int64_t rows, int64_t K, int group,
                                  __half* w) {
  const int64_t nb = rows * K / 2;   // one byte = two codes
  const int64_t ng = K / group;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nb;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = 2 * i, row = e / K, col = e % K;   // col even, col + 1 in the same group
    const int64_t gi = row * ng + col / group;
    const float s = __half2float(scale[gi]);
    const int z = zero[gi];
    const int b = packed[i];
    reinterpret_cast<__half2*>(w)[i] =
        __floats2half2_rn(s * (float)((b & 15) - z), s * (float)((b >> 4) - z));
  }
}

}  // namespace

cudaError_t launch_dequant(int fmt, const void* q, const void* scale, const void* zero,
                           int64_t rows, int64_t K, int group, __half* w, int num_sms,
                           cudaStream_t s) {
  const int threads = 256, blocks = 4 * num_sms;
  if (fmt == 1) {
    dequant_i8_kernel<<<blocks, threads, 0, s>>>(static_cast<const int8_t*>(q),
                                                 static_cast<const __half*>(scale), rows, K, w);
  } else if (fmt == 2) {
    dequant_u4_kernel<<<blocks, threads, 0, s>>>(static_cast<const uint8_t*>(q),
                                                 static_cast<const __half*>(scale),
                                                 static_cast<const uint8_t*>(zero), rows, K,
                                                 group, w);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace blk
