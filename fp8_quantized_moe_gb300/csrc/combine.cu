// Ragged gather-reduce ("Quantize activations before EP all gather":
// ragged_gather_reduce un-permutes the expert outputs and sums the top-k rows
// of every token weighted by its router probabilities).
//
//   out[t, :] = bf16( sum_{j < k} w[t, j] * rows[pos[t*k + j], :] )
//
// HBM-bound: one warp per token; per pass each lane loads two 16-byte vectors
// (8 bf16 each) from every source row, the loads of up to KB rows (KB >= k up
// to 8) issued before any of them is accumulated (so that a pass costs one
// memory latency, not k: with few tokens, as in a prefill chunk, the warps
// cannot hide a chain of them; KB fits k so that small k keeps its registers
// and occupancy), accumulates in fp32 in ascending j, and writes 8 bf16 a
// vector.
#include "common.cuh"

namespace moe {
namespace {

__device__ unsigned int g_err;

constexpr int kMaxK = 32;

template <int KB>
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* rows, const int32_t* pos,
                                                      const float* weights, int64_t T, int k, int64_t D,
                                                      uint16_t* out) {
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const int64_t R = T * k;
  int my_pos = 0;
  float my_w = 0.0f;
  if (lane < k) {
    const int p = __ldg(pos + t * k + lane);
    my_pos = (p >= 0 && p < R) ? p : -1;
    if (my_pos < 0) raise_error(&g_err, MOE_DEVERR_BAD_POSITION);  // a corrupted permutation
    my_w = weights ? __ldg(weights + t * k + lane) : 1.0f;
  }
  const int64_t nvec = D / 8;
  constexpr int kBatch = KB;  // source rows whose loads are in flight together
  // every lane runs every pass (the row positions and weights are broadcast
  // by shuffles from the lanes that loaded them), with its own vectors masked
  for (int64_t vbase = 0; vbase < nvec; vbase += 64) {
    const int64_t v0 = vbase + lane;
    float acc[2][8];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[u][c] = 0.0f;
    for (int j0 = 0; j0 < k; j0 += kBatch) {
      uint4 d[kBatch][2];
      float w[kBatch];
      bool ok[kBatch];
#pragma unroll
      for (int jj = 0; jj < kBatch; ++jj) {  // every load of the batch first
        const int j = j0 + jj;
        const int p = __shfl_sync(0xffffffffu, my_pos, j & 31);
        w[jj] = __shfl_sync(0xffffffffu, my_w, j & 31);
        ok[jj] = j < k && p >= 0;
        const uint16_t* src = rows + static_cast<int64_t>(ok[jj] ? p : 0) * D;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int64_t v = v0 + 32 * u;
          d[jj][u] = (ok[jj] && v < nvec) ? __ldg(reinterpret_cast<const uint4*>(src + 8 * v)) : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int jj = 0; jj < kBatch; ++jj) {  // then the sums, in ascending j
        if (!ok[jj]) continue;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint32_t wd[4] = {d[jj][u].x, d[jj][u].y, d[jj][u].z, d[jj][u].w};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            acc[u][2 * c] = __fmaf_rn(w[jj], bf16lo(wd[c]), acc[u][2 * c]);
            acc[u][2 * c + 1] = __fmaf_rn(w[jj], bf16hi(wd[c]), acc[u][2 * c + 1]);
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int64_t v = v0 + 32 * u;
      if (v < nvec) {
        uint4 o;
        o.x = pack_bf16x2(acc[u][0], acc[u][1]);
        o.y = pack_bf16x2(acc[u][2], acc[u][3]);
        o.z = pack_bf16x2(acc[u][4], acc[u][5]);
        o.w = pack_bf16x2(acc[u][6], acc[u][7]);
        *reinterpret_cast<uint4*>(out + t * D + 8 * v) = o;
      }
    }
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" __attribute__((visibility("hidden"))) cudaError_t moe_detail_take_error_combine(unsigned int* out) {
  unsigned int v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_err, sizeof(v));
  if (e == cudaSuccess && v) e = cudaMemcpyToSymbol(g_err, &z, sizeof(z));
  *out = v;
  return e;
}

extern "C" moe_status ragged_gather_reduce(const uint16_t* rows, const int32_t* pos, const float* weights, int64_t T,
                                           int k, int64_t D, uint16_t* out, moe_stream_t stream) {
  MOE_HOST_CHECK(rows && pos && out && T >= 0 && k > 0 && k <= kMaxK && D > 0 && D % 8 == 0, MOE_ERR_INVALID_ARG);
  // T * k < 2^31, tested without forming the product of an unchecked T
  MOE_HOST_CHECK(T <= ((1ll << 31) - 1) / k && aligned16(rows) && aligned16(out), MOE_ERR_INVALID_ARG);
  if (T == 0) return MOE_OK;
  const unsigned grid = static_cast<unsigned>((T + 7) / 8);
  cudaStream_t st = as_stream(stream);
  if (k <= 2)
    combine_kernel<2><<<grid, 256, 0, st>>>(rows, pos, weights, T, k, D, out);
  else if (k <= 4)
    combine_kernel<4><<<grid, 256, 0, st>>>(rows, pos, weights, T, k, D, out);
  else
    combine_kernel<8><<<grid, 256, 0, st>>>(rows, pos, weights, T, k, D, out);
  MOE_CUDA_TRY(cudaGetLastError());
  return MOE_OK;
}
