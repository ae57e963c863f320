// Router backward helpers ("Support quantization for tokamax gmm v2", table 1:
// the gate kernel's gradient grad_gate-kernel and the state gradient
// state_grad are measured beside the expert weights' gradients).
//
//   dw[t, j]         = <G[t], o[pos[t k + j]]>       (the combine's adjoint in w)
//   dlogits[t, i]    = bf16( p_i (g_i - s) ),  s = sum_j p[id_j] dw[t, j],
//                      g_i = dw[t, j] where i = id_j (else 0)
// with p the fp32 softmax of the row's logits taken exactly as the router's
// forward takes it (max, e_i = exp(l_i - m), Z summed in ascending i,
// p_i = e_i / Z).  The two gate gradients are dense bf16 contractions run by
// the tcgen05 kernels; this file lays out their operands (transposed and
// zero-padded so that every row pitch is a multiple of 16 bytes).
#include "common.cuh"

namespace moe {
namespace {

// One warp per token: the k dot products of length D, 16-byte loads, fp32
// partial sums reduced across the warp.
__global__ void __launch_bounds__(256) router_dw_kernel(const uint16_t* G, const uint16_t* o, const int32_t* pos,
                                                        int64_t T, int k, int64_t D, float* dw) {
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const uint4* g = reinterpret_cast<const uint4*>(G + t * D);
  const int64_t nvec = D / 8;
  for (int j = 0; j < k; ++j) {
    const int64_t r = __ldg(pos + t * k + j);
    const uint4* src = reinterpret_cast<const uint4*>(o + r * D);
    float acc = 0.0f;
    for (int64_t v = lane; v < nvec; v += 32) {
      const uint4 a = __ldg(g + v), b = __ldg(src + v);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        acc = __fmaf_rn(bf16lo(aw[c]), bf16lo(bw[c]), acc);
        acc = __fmaf_rn(bf16hi(aw[c]), bf16hi(bw[c]), acc);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) dw[t * k + j] = acc;
  }
}

// One thread per token row t < Tp (rows T..Tp-1 only zero the padding of the
// transposed copy).  Writes dlogits [T, E], the same values into a [T, Ep]
// copy whose columns E..Ep-1 are zero, and the transpose [Ep, Tp] (zero past
// T and past E).
__global__ void __launch_bounds__(128) router_dlogits_kernel(const float* logits, const int32_t* ids, const float* dw,
                                                             int64_t T, int E, int k, int Ep, int64_t Tp,
                                                             uint16_t* dl, uint16_t* dl_pad, uint16_t* dlT) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= Tp) return;
  if (t >= T) {
    for (int i = 0; i < Ep; ++i) dlT[static_cast<int64_t>(i) * Tp + t] = 0;
    return;
  }
  const float* l = logits + t * E;
  float m = -INFINITY;
  for (int i = 0; i < E; ++i) m = fmaxf(m, l[i]);
  float z = 0.0f;
  for (int i = 0; i < E; ++i) z = __fadd_rn(z, exp_f32(__fsub_rn(l[i], m)));
  float s = 0.0f;
  for (int j = 0; j < k; ++j) {
    const int e = __ldg(ids + t * k + j);
    const float wj = __fdiv_rn(exp_f32(__fsub_rn(l[e], m)), z);
    s = __fadd_rn(s, __fmul_rn(wj, __ldg(dw + t * k + j)));
  }
  for (int i = 0; i < Ep; ++i) {
    uint16_t b = 0;
    if (i < E) {
      float g = 0.0f;
      for (int j = 0; j < k; ++j)
        if (__ldg(ids + t * k + j) == i) g = __ldg(dw + t * k + j);
      const float pi = __fdiv_rn(exp_f32(__fsub_rn(l[i], m)), z);
      b = static_cast<uint16_t>(pack_bf16x2(__fmul_rn(pi, __fsub_rn(g, s)), 0.0f) & 0xFFFFu);
      dl[t * E + i] = b;
    }
    dl_pad[t * Ep + i] = b;
    dlT[static_cast<int64_t>(i) * Tp + t] = b;
  }
}

// src [R, C] -> dst [C, Rp] (2-byte elements), columns R..Rp-1 of dst zero.
// 32 x 32 tiles through shared memory (one padded column against bank
// conflicts); a block of 32 x 8 threads moves one tile.
__global__ void __launch_bounds__(256) transpose_u16_kernel(const uint16_t* src, int64_t R, int64_t C, uint16_t* dst,
                                                            int64_t Rp) {
  __shared__ uint16_t tile[32][33];
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 32, c0 = static_cast<int64_t>(blockIdx.x) * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int i = ty; i < 32; i += 8) {
    const int64_t r = r0 + i, c = c0 + tx;
    tile[i][tx] = (r < R && c < C) ? src[r * C + c] : static_cast<uint16_t>(0);
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int64_t c = c0 + i, r = r0 + tx;
    if (c < C && r < Rp) dst[c * Rp + r] = tile[tx][i];
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" __attribute__((visibility("hidden"))) cudaError_t moe_detail_router_dw(const uint16_t* G, const uint16_t* o,
                                                                                  const int32_t* pos, int64_t T, int k,
                                                                                  int64_t D, float* dw,
                                                                                  cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  router_dw_kernel<<<static_cast<unsigned>((T + 7) / 8), 256, 0, st>>>(G, o, pos, T, k, D, dw);
  return cudaGetLastError();
}

extern "C" __attribute__((visibility("hidden"))) cudaError_t moe_detail_router_dlogits(
    const float* logits, const int32_t* ids, const float* dw, int64_t T, int E, int k, int Ep, int64_t Tp,
    uint16_t* dl, uint16_t* dl_pad, uint16_t* dlT, cudaStream_t st) {
  if (Tp == 0) return cudaSuccess;
  router_dlogits_kernel<<<static_cast<unsigned>((Tp + 127) / 128), 128, 0, st>>>(logits, ids, dw, T, E, k, Ep, Tp, dl,
                                                                                 dl_pad, dlT);
  return cudaGetLastError();
}

extern "C" __attribute__((visibility("hidden"))) cudaError_t moe_detail_transpose_u16(const uint16_t* src, int64_t R,
                                                                                      int64_t C, uint16_t* dst,
                                                                                      int64_t Rp, cudaStream_t st) {
  if (Rp == 0 || C == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((C + 31) / 32), static_cast<unsigned>((Rp + 31) / 32));
  transpose_u16_kernel<<<grid, 256, 0, st>>>(src, R, C, dst, Rp);
  return cudaGetLastError();
}
