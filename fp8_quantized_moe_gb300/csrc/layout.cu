// Batched byte transpose for weight layout preparation: src [B, R, C] ->
// dst [B, C, R].  64 x 64 byte tiles staged through shared memory; 16-byte
// global loads and stores.
#include "common.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) transpose_u8_kernel(const uint8_t* src, int64_t R, int64_t C, uint8_t* dst) {
  __shared__ __align__(16) uint8_t tile[64][80];
  const int64_t b = blockIdx.z;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 64, c0 = static_cast<int64_t>(blockIdx.x) * 64;
  const uint8_t* s = src + b * R * C;
  uint8_t* d = dst + b * R * C;
  {
    const int rr = threadIdx.x >> 2, part = threadIdx.x & 3;
    const int64_t r = r0 + rr, c = c0 + part * 16;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < R && c < C) v = __ldg(reinterpret_cast<const uint4*>(s + r * C + c));
    *reinterpret_cast<uint4*>(&tile[rr][part * 16]) = v;
  }
  __syncthreads();
  {
    const int cc = threadIdx.x >> 2, part = threadIdx.x & 3;
    const int64_t c = c0 + cc, r = r0 + part * 16;
    if (c < C && r < R) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int rb = part * 16 + q * 4;
        w[q] = static_cast<uint32_t>(tile[rb][cc]) | (static_cast<uint32_t>(tile[rb + 1][cc]) << 8) |
               (static_cast<uint32_t>(tile[rb + 2][cc]) << 16) | (static_cast<uint32_t>(tile[rb + 3][cc]) << 24);
      }
      *reinterpret_cast<uint4*>(d + c * R + r) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_transpose_u8(const uint8_t* src, int64_t B, int64_t R, int64_t C, uint8_t* dst,
                                       moe_stream_t stream) {
  MOE_HOST_CHECK(src && dst && B > 0 && R > 0 && C > 0 && R % 16 == 0 && C % 16 == 0, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(B < 65536 && (R + 63) / 64 < 65536 && moe::aligned16(src) && moe::aligned16(dst),
                 MOE_ERR_INVALID_ARG);
  dim3 grid(static_cast<unsigned>((C + 63) / 64), static_cast<unsigned>((R + 63) / 64), static_cast<unsigned>(B));
  moe::transpose_u8_kernel<<<grid, 256, 0, moe::as_stream(stream)>>>(src, R, C, dst);
  MOE_CUDA_TRY(cudaGetLastError());
  return MOE_OK;
}
