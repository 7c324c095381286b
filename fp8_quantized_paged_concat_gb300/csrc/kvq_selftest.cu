// kvq_selftest.cu -- runs the device converters of kvq_device.cuh over a
// range of float32 bit patterns so that tests can compare them, pattern by
// pattern, with an independent implementation.  Not on the cache path.
#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

__global__ void __launch_bounds__(256) selftest_convert_kernel(
    uint32_t first_bits, int64_t count, uint8_t* e4m3_lo, uint8_t* e4m3_hi, uint8_t* e2m1_lo,
    uint8_t* e2m1_hi, uint16_t* bf16_out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
       i += stride) {
    const float f = __uint_as_float(first_bits + static_cast<uint32_t>(i));
    if (e4m3_lo) e4m3_lo[i] = static_cast<uint8_t>(cvt_e4m3x2(f, 0.0f) & 0xffu);
    if (e4m3_hi) e4m3_hi[i] = static_cast<uint8_t>(cvt_e4m3x2(0.0f, f) >> 8);
    if (e2m1_lo) e2m1_lo[i] = static_cast<uint8_t>(cvt_e2m1x2(f, 0.0f) & 0xfu);
    if (e2m1_hi) e2m1_hi[i] = static_cast<uint8_t>(cvt_e2m1x2(0.0f, f) >> 4);
    if (bf16_out) bf16_out[i] = static_cast<uint16_t>(pack_bf16x2(f, 0.0f) & 0xffffu);
  }
}

}  // namespace

cudaError_t launch_selftest_convert(uint32_t first_bits, int64_t count, uint8_t* e4m3_lo,
                                    uint8_t* e4m3_hi, uint8_t* e2m1_lo, uint8_t* e2m1_hi,
                                    uint16_t* bf16_out, int num_sms, cudaStream_t stream) {
  int64_t blocks = (count + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;   // grid-stride beyond 8 CTAs per SM
  if (blocks > cap) blocks = cap;
  selftest_convert_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      first_bits, count, e4m3_lo, e4m3_hi, e2m1_lo, e2m1_hi, bf16_out);
  return cudaGetLastError();
}

}  // namespace kvq
