// Ragged sort of the (token, expert) pairs by routed expert, plus the gather
// of the quantised rows and (per-token) scales -- "Quantize activations
// before EP all gather": the activations are quantised first, so the sort
// moves fp8 rows, and the scale rows are gathered only when the scale is per
// token.
//
// Stable counting sort over the flat pairs i = t*k + j, keyed by expert id:
//   1. hist:    each CTA owns a chunk of 2048 pairs (8 warps x 256); per-warp
//               histograms in shared memory, chunk totals to the workspace.
//   2. scan:    one CTA: per expert, prefix over chunks; across experts, a
//               block-wide exclusive scan -> group_sizes, group_offsets and
//               the first output slot of every (chunk, expert).
//   3. scatter: each warp walks its 256 pairs in index order, 32 at a time;
//               __match_any_sync ranks equal ids inside a round, per-warp
//               running counters carry the rank across rounds -> stable.
//   4. gather:  one warp per token reads its fp8 row once (16-byte loads) and
//               writes it to the k sorted positions; scales alongside.
// Small problems (up to 32768 pairs and 64 experts) run steps 1-3 in one CTA
// instead of three launches (sort_small_kernel); with more experts a round of
// 32 pairs holds more distinct ids and the multi-CTA path is faster
// (measured: 16384 pairs over 8 experts 7 us faster in one CTA, over 128
// experts 4 us slower).
#include "common.cuh"

namespace moe {
namespace {

__device__ unsigned int g_err;

constexpr int kWarps = 8;
constexpr int kPerWarp = 256;
constexpr int kChunk = kWarps * kPerWarp;  // 2048 pairs per CTA
constexpr int kMaxE = 1024;

__device__ __forceinline__ int load_id(const int32_t* ids, int64_t i, int64_t R, int E, bool& bad) {
  if (i >= R) return -1;
  const int e = __ldg(ids + i);
  if (e < 0 || e >= E) {
    bad = true;
    return -1;
  }
  return e;
}

constexpr int kRounds = kPerWarp / 32;  // rounds of 32 pairs per warp

// Per-warp histograms of the chunk; hist is [kWarps][E] in shared memory.
// The ids of the warp's kRounds rounds are loaded together (one memory
// latency, not kRounds) and returned in ev for the scatter.
__device__ __forceinline__ void chunk_hist(const int32_t* ids, int64_t R, int E, int* hist, int (&ev)[kRounds]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kWarps * E; i += blockDim.x) hist[i] = 0;
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kChunk + warp * kPerWarp;
  bool bad = false;
#pragma unroll
  for (int r = 0; r < kRounds; ++r) ev[r] = load_id(ids, base + r * 32 + lane, R, E, bad);
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kRounds; ++r)
    if (ev[r] >= 0) atomicAdd(&hist[warp * E + ev[r]], 1);
  if (bad) raise_error(&g_err, MOE_DEVERR_BAD_EXPERT_ID);
  __syncthreads();
}

__global__ void __launch_bounds__(256) sort_hist_kernel(const int32_t* ids, int64_t R, int E, int* chunk_counts) {
  extern __shared__ int hist[];
  int ev[kRounds];
  chunk_hist(ids, R, E, hist, ev);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int s = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += hist[w * E + e];
    chunk_counts[static_cast<int64_t>(blockIdx.x) * E + e] = s;
  }
}

// Exclusive scan of `v` over the 1024 threads of the CTA (thread order).
__device__ __forceinline__ int block_exclusive_scan_1024(int v, int* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = warp_sums[lane];
    int inc2 = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc2, o);
      if (lane >= o) inc2 += t;
    }
    warp_sums[lane] = inc2 - w;
  }
  __syncthreads();
  return incl - v + warp_sums[warp];
}

// One CTA of 1024 threads; thread e owns expert e.
__global__ void __launch_bounds__(1024) sort_scan_kernel(int* chunk_counts, int nchunks, int E,
                                                         int32_t* group_sizes, int32_t* group_offsets) {
  __shared__ int warp_sums[32];
  const int e = threadIdx.x;
  int total = 0;
  if (e < E) {
    for (int c = 0; c < nchunks; ++c) {
      const int v = chunk_counts[static_cast<int64_t>(c) * E + e];
      chunk_counts[static_cast<int64_t>(c) * E + e] = total;  // exclusive within the expert
      total += v;
    }
  }
  // block-wide exclusive scan of total over experts
  const int excl = block_exclusive_scan_1024(total, warp_sums);
  if (e < E) {
    group_sizes[e] = total;
    group_offsets[e] = excl;
    if (e == E - 1) group_offsets[E] = excl + total;
    for (int c = 0; c < nchunks; ++c) chunk_counts[static_cast<int64_t>(c) * E + e] += excl;
  }
}

__global__ void __launch_bounds__(256) sort_scatter_kernel(const int32_t* ids, int64_t R, int E,
                                                           const int* chunk_counts, int32_t* sorted_src,
                                                           int32_t* pos) {
  extern __shared__ int hist[];  // [kWarps][E] counts, then running slots
  int ev[kRounds];
  chunk_hist(ids, R, E, hist, ev);
  // hist[w][e] <- first slot of warp w's pairs of expert e
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = chunk_counts[static_cast<int64_t>(blockIdx.x) * E + e];
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* slot = hist + warp * E;
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kChunk + warp * kPerWarp;
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int64_t i = base + r * 32 + lane;
    const int e = ev[r];
    const unsigned valid = __ballot_sync(0xffffffffu, e >= 0);
    if (e >= 0) {
      const unsigned peers = __match_any_sync(valid, e);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int p = slot[e] + rank;
      sorted_src[p] = static_cast<int32_t>(i);
      pos[i] = p;
      __syncwarp(valid);
      if (rank == 0) slot[e] += __popc(peers);
    }
    __syncwarp();
  }
}

// Steps 1-3 for a small problem in one CTA of 1024 threads (R <= kSmallMaxR
// pairs, E <= kSmallMaxE): warp w owns the contiguous pairs [w per, (w + 1)
// per) and walks them 32 at a time, the loads of eight rounds in flight
// together; the scan runs in shared memory, and sorted_src is assembled there
// and written out in order (its slots are scattered across the experts, pos
// is written coalesced where it is made).  The order is the same stable order
// as the multi-CTA path's (by expert, then by pair index).
constexpr int kSmallWarps = 32;
constexpr int kSmallMaxE = 64;
constexpr int64_t kSmallMaxR = 32768;
constexpr int kSmallBatch = 8;  // rounds whose id loads are in flight together
__global__ void __launch_bounds__(1024) sort_small_kernel(const int32_t* ids, int64_t R, int E, int32_t* sorted_src,
                                                          int32_t* pos, int32_t* group_sizes,
                                                          int32_t* group_offsets) {
  extern __shared__ int sm_small[];
  int* hist = sm_small;                           // [warp][expert]: counts, then first slots
  int* stage = sm_small + kSmallWarps * E;        // sorted_src, assembled here [R]
  __shared__ int warp_sums[32];
  __shared__ int nvalid;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // rounds of 32 pairs per warp
  const int rounds = static_cast<int>((R + kSmallWarps * 32 - 1) / (kSmallWarps * 32));
  for (int i = threadIdx.x; i < kSmallWarps * E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int64_t base = static_cast<int64_t>(warp) * rounds * 32;
  bool bad = false;
  for (int r0 = 0; r0 < rounds; r0 += kSmallBatch) {
    int eb[kSmallBatch];
#pragma unroll
    for (int b = 0; b < kSmallBatch; ++b)
      eb[b] = r0 + b < rounds ? load_id(ids, base + (r0 + b) * 32 + lane, R, E, bad) : -1;
#pragma unroll
    for (int b = 0; b < kSmallBatch; ++b)
      if (eb[b] >= 0) atomicAdd(&hist[warp * E + eb[b]], 1);
  }
  if (bad) raise_error(&g_err, MOE_DEVERR_BAD_EXPERT_ID);
  __syncthreads();
  // thread e: expert e's counts over the warps -> exclusive within the
  // expert; the experts' totals -> group sizes and offsets
  const int e = threadIdx.x;
  int total = 0;
  if (e < E) {
    for (int w = 0; w < kSmallWarps; ++w) {
      const int v = hist[w * E + e];
      hist[w * E + e] = total;
      total += v;
    }
  }
  const int excl = block_exclusive_scan_1024(total, warp_sums);
  if (e < E) {
    group_sizes[e] = total;
    group_offsets[e] = excl;
    if (e == E - 1) {
      group_offsets[E] = excl + total;
      nvalid = excl + total;
    }
    for (int w = 0; w < kSmallWarps; ++w) hist[w * E + e] += excl;
  }
  __syncthreads();
  int* slot = hist + warp * E;
  for (int r0 = 0; r0 < rounds; r0 += kSmallBatch) {
    int eb[kSmallBatch];
    bool unused = false;
#pragma unroll
    for (int b = 0; b < kSmallBatch; ++b)
      eb[b] = r0 + b < rounds ? load_id(ids, base + (r0 + b) * 32 + lane, R, E, unused) : -1;
#pragma unroll
    for (int b = 0; b < kSmallBatch; ++b) {
      if (r0 + b >= rounds) break;  // the same for every lane of the warp
      const int64_t i = base + (r0 + b) * 32 + lane;
      const unsigned valid = __ballot_sync(0xffffffffu, eb[b] >= 0);
      if (eb[b] >= 0) {
        const unsigned peers = __match_any_sync(valid, eb[b]);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        const int p = slot[eb[b]] + rank;
        stage[p] = static_cast<int>(i);
        pos[i] = p;
        __syncwarp(valid);
        if (rank == 0) slot[eb[b]] += __popc(peers);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  for (int p = threadIdx.x; p < nvalid; p += blockDim.x) sorted_src[p] = stage[p];
}

// One warp per token: read the fp8 row once, write it to its k slots.
template <int MODE>
__global__ void __launch_bounds__(256) sort_gather_kernel(const uint8_t* x_q, const float* x_scale, int64_t T,
                                                          int k, int64_t D, const int32_t* pos, uint8_t* xs_q,
                                                          float* xs_scale) {
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const int64_t R = T * k;
  int my_pos = -1;
  if (lane < k) {
    my_pos = pos[t * k + lane];
    if (my_pos < 0 || my_pos >= R) my_pos = -1;
  }
  const uint8_t* src = x_q + t * D;
  constexpr int CH = 8;  // 16-byte vectors per lane per pass (4 KB per warp)
  for (int64_t b0 = 0; b0 < D; b0 += 32 * 16 * CH) {
    uint4 v[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int64_t off = b0 + (static_cast<int64_t>(c) * 32 + lane) * 16;
      if (off < D) v[c] = __ldg(reinterpret_cast<const uint4*>(src + off));
    }
    for (int j = 0; j < k; ++j) {
      const int p = __shfl_sync(0xffffffffu, my_pos, j);
      if (p < 0) continue;
      uint8_t* dst = xs_q + static_cast<int64_t>(p) * D;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int64_t off = b0 + (static_cast<int64_t>(c) * 32 + lane) * 16;
        if (off < D) *reinterpret_cast<uint4*>(dst + off) = v[c];
      }
    }
  }
  if (MODE == MOE_SCALE_PER_ROW) {
    if (my_pos >= 0) xs_scale[my_pos] = __ldg(x_scale + t);
  } else if (MODE == MOE_SCALE_PER_ROW_BLOCK128) {
    const int64_t nb = (D + 127) / 128;
    for (int j = 0; j < k; ++j) {
      const int p = __shfl_sync(0xffffffffu, my_pos, j);
      if (p < 0) continue;
      for (int64_t b = lane; b < nb; b += 32) xs_scale[static_cast<int64_t>(p) * nb + b] = __ldg(x_scale + t * nb + b);
    }
  }
}

int64_t num_chunks(int64_t R) { return (R + kChunk - 1) / kChunk; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" __attribute__((visibility("hidden"))) cudaError_t moe_detail_take_error_sort(unsigned int* out) {
  unsigned int v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_err, sizeof(v));
  if (e == cudaSuccess && v) e = cudaMemcpyToSymbol(g_err, &z, sizeof(z));
  *out = v;
  return e;
}

namespace moe {
namespace {
// T * k < 2^31 (the pair indices are int32), tested without forming the
// product of an unchecked T.
bool pairs_fit(int64_t T, int k) { return T >= 0 && k > 0 && T <= ((1ll << 31) - 1) / k; }
}  // namespace
}  // namespace moe

extern "C" size_t moe_ragged_sort_workspace_bytes(int64_t T, int k, int E) {
  if (!moe::pairs_fit(T, k) || E <= 0) return 0;
  const int64_t nc = num_chunks(T * k);
  return static_cast<size_t>((nc > 0 ? nc : 1) * E) * sizeof(int);
}

namespace moe {
namespace {
// Steps of the sort that produce the indices: histogram, scan, stable
// scatter.  `counts` is the caller's workspace.
moe_status sort_indices(const int32_t* topk_ids, int64_t T, int k, int E, int32_t* sorted_src, int32_t* pos,
                        int32_t* group_sizes, int32_t* group_offsets, int* counts, cudaStream_t st) {
  const int64_t R = T * k;
  if (R > 0 && E <= kSmallMaxE && R <= kSmallMaxR) {  // one CTA, one launch
    const size_t smem = sizeof(int) * (static_cast<size_t>(kSmallWarps) * E + static_cast<size_t>(R));
    MOE_CUDA_TRY(cudaFuncSetAttribute(sort_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(sizeof(int) * (kSmallWarps * kSmallMaxE + kSmallMaxR))));
    sort_small_kernel<<<1, 1024, smem, st>>>(topk_ids, R, E, sorted_src, pos, group_sizes, group_offsets);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
  }
  const int64_t nc = num_chunks(R);
  const size_t hist_smem = sizeof(int) * kWarps * E;
  if (nc > 0) {
    if (hist_smem > 48 * 1024) {
      MOE_CUDA_TRY(cudaFuncSetAttribute(sort_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(hist_smem)));
      MOE_CUDA_TRY(cudaFuncSetAttribute(sort_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(hist_smem)));
    }
    sort_hist_kernel<<<static_cast<unsigned>(nc), 256, hist_smem, st>>>(topk_ids, R, E, counts);
    MOE_CUDA_TRY(cudaGetLastError());
  }
  sort_scan_kernel<<<1, 1024, 0, st>>>(counts, static_cast<int>(nc), E, group_sizes, group_offsets);
  MOE_CUDA_TRY(cudaGetLastError());
  if (nc == 0) return MOE_OK;
  sort_scatter_kernel<<<static_cast<unsigned>(nc), 256, hist_smem, st>>>(topk_ids, R, E, counts, sorted_src, pos);
  MOE_CUDA_TRY(cudaGetLastError());
  return MOE_OK;
}
}  // namespace
}  // namespace moe

extern "C" moe_status moe_ragged_sort(const int32_t* topk_ids, int64_t T, int k, int E, const uint8_t* x_q,
                                      const float* x_scale, int64_t D, moe_scale_mode mode, int32_t* sorted_src,
                                      int32_t* pos, int32_t* group_sizes, int32_t* group_offsets, uint8_t* xs_q,
                                      float* xs_scale, void* workspace, size_t workspace_bytes,
                                      moe_stream_t stream) {
  MOE_HOST_CHECK(topk_ids && x_q && sorted_src && pos && group_sizes && group_offsets && xs_q && workspace,
                 MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(T >= 0 && k > 0 && k <= 32 && E > 0 && E <= kMaxE && D > 0 && D % 16 == 0, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(pairs_fit(T, k), MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(aligned16(x_q) && aligned16(xs_q) && (reinterpret_cast<uintptr_t>(workspace) & 3) == 0,
                 MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(workspace_bytes >= moe_ragged_sort_workspace_bytes(T, k, E), MOE_ERR_INVALID_ARG);
  if (mode == MOE_SCALE_PER_ROW || mode == MOE_SCALE_PER_ROW_BLOCK128) {
    MOE_HOST_CHECK(x_scale && xs_scale, MOE_ERR_INVALID_ARG);
  } else {
    MOE_HOST_CHECK(mode == MOE_SCALE_PER_TENSOR, MOE_ERR_INVALID_ARG);
  }
  cudaStream_t st = as_stream(stream);
  moe_status stt = sort_indices(topk_ids, T, k, E, sorted_src, pos, group_sizes, group_offsets,
                                static_cast<int*>(workspace), st);
  if (stt != MOE_OK || T * k == 0) return stt;
  const unsigned gblocks = static_cast<unsigned>((T + 7) / 8);
  if (mode == MOE_SCALE_PER_ROW)
    sort_gather_kernel<MOE_SCALE_PER_ROW><<<gblocks, 256, 0, st>>>(x_q, x_scale, T, k, D, pos, xs_q, xs_scale);
  else if (mode == MOE_SCALE_PER_ROW_BLOCK128)
    sort_gather_kernel<MOE_SCALE_PER_ROW_BLOCK128>
        <<<gblocks, 256, 0, st>>>(x_q, x_scale, T, k, D, pos, xs_q, xs_scale);
  else
    sort_gather_kernel<MOE_SCALE_PER_TENSOR><<<gblocks, 256, 0, st>>>(x_q, x_scale, T, k, D, pos, xs_q, xs_scale);
  MOE_CUDA_TRY(cudaGetLastError());
  return MOE_OK;
}

extern "C" __attribute__((visibility("hidden"))) moe_status moe_detail_quantize_gather(
    const uint16_t* x, const int32_t* pos, int64_t T, int k, int64_t D, moe_scale_mode mode, const float* static_scale,
    uint8_t* xs_q, float* xs_scale, cudaStream_t st);

extern "C" moe_status moe_quantize_sort(const uint16_t* x, const int32_t* topk_ids, int64_t T, int k, int E, int64_t D,
                                        moe_scale_mode mode, const float* static_scale, int32_t* sorted_src,
                                        int32_t* pos, int32_t* group_sizes, int32_t* group_offsets, uint8_t* xs_q,
                                        float* xs_scale, void* workspace, size_t workspace_bytes,
                                        moe_stream_t stream) {
  MOE_HOST_CHECK(x && topk_ids && sorted_src && pos && group_sizes && group_offsets && xs_q && workspace,
                 MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(T >= 0 && k > 0 && k <= 32 && E > 0 && E <= kMaxE && D > 0 && D % 16 == 0, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(pairs_fit(T, k), MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(aligned16(x) && aligned16(xs_q) && (reinterpret_cast<uintptr_t>(workspace) & 3) == 0,
                 MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(workspace_bytes >= moe_ragged_sort_workspace_bytes(T, k, E), MOE_ERR_INVALID_ARG);
  if (mode == MOE_SCALE_PER_ROW || mode == MOE_SCALE_PER_ROW_BLOCK128) {
    MOE_HOST_CHECK(xs_scale != nullptr && aligned16(xs_scale), MOE_ERR_INVALID_ARG);
  } else {
    MOE_HOST_CHECK(mode == MOE_SCALE_PER_TENSOR && static_scale, MOE_ERR_INVALID_ARG);
  }
  cudaStream_t st = as_stream(stream);
  moe_status stt = sort_indices(topk_ids, T, k, E, sorted_src, pos, group_sizes, group_offsets,
                                static_cast<int*>(workspace), st);
  if (stt != MOE_OK || T * k == 0) return stt;
  return moe_detail_quantize_gather(x, pos, T, k, D, mode, static_scale, xs_q, xs_scale, st);
}

extern "C" __attribute__((visibility("hidden"))) moe_status moe_detail_quantize_gather_mx(
    const uint16_t* x, const int32_t* pos, int64_t T, int k, int64_t D, uint8_t* xs_q, uint8_t* xs_sf,
    cudaStream_t st);

// MXFP8 form of moe_quantize_sort: the codes and the E8M0 codes of each token
// row go to its k sorted rows.
extern "C" moe_status moe_quantize_sort_mx(const uint16_t* x, const int32_t* topk_ids, int64_t T, int k, int E,
                                           int64_t D, int32_t* sorted_src, int32_t* pos, int32_t* group_sizes,
                                           int32_t* group_offsets, uint8_t* xs_q, uint8_t* xs_sf, void* workspace,
                                           size_t workspace_bytes, moe_stream_t stream) {
  MOE_HOST_CHECK(x && topk_ids && sorted_src && pos && group_sizes && group_offsets && xs_q && xs_sf && workspace,
                 MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(T >= 0 && k > 0 && k <= 32 && E > 0 && E <= kMaxE && D > 0 && D % 128 == 0, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(pairs_fit(T, k), MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(aligned16(x) && aligned16(xs_q) && (reinterpret_cast<uintptr_t>(workspace) & 3) == 0,
                 MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(workspace_bytes >= moe_ragged_sort_workspace_bytes(T, k, E), MOE_ERR_INVALID_ARG);
  cudaStream_t st = as_stream(stream);
  moe_status stt = sort_indices(topk_ids, T, k, E, sorted_src, pos, group_sizes, group_offsets,
                                static_cast<int*>(workspace), st);
  if (stt != MOE_OK || T * k == 0) return stt;
  return moe_detail_quantize_gather_mx(x, pos, T, k, D, xs_q, xs_sf, st);
}

// ---------------------------------------------------------------------------
// moe_ragged_sort_noalloc: the same sort for callers that cannot allocate
// device memory.  Its scratch (the per-(chunk, expert) counts) lives in a
// fixed file-scope device array; every GPU that loads this library holds it
// until the process exits.  Host code cannot pass `g_sort_scratch` itself to
// a kernel (in host code the name denotes a host-side shadow, not a device
// address), so the device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call.
// ---------------------------------------------------------------------------
#include <mutex>

namespace moe {
namespace {

constexpr size_t kNoAllocScratchBytes = MOE_RAGGED_SORT_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) int g_sort_scratch[kNoAllocScratchBytes / sizeof(int)];

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace
}  // namespace moe

extern "C" moe_status moe_ragged_sort_noalloc(const int32_t* topk_ids, int64_t T, int k, int E, const uint8_t* x_q,
                                              const float* x_scale, int64_t D, moe_scale_mode mode,
                                              int32_t* sorted_src, int32_t* pos, int32_t* group_sizes,
                                              int32_t* group_offsets, uint8_t* xs_q, float* xs_scale,
                                              moe_stream_t stream) {
  if (!moe::pairs_fit(T, k) || E <= 0) return MOE_ERR_INVALID_ARG;
  // the counts need nchunks * E ints; larger problems do not fit the array
  if (moe_ragged_sort_workspace_bytes(T, k, E) > moe::kNoAllocScratchBytes) return MOE_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= moe::kMaxDevices) return MOE_ERR_CUDA;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(moe::g_scratch_mu);
    if (!moe::g_scratch_addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, moe::g_sort_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
      moe::g_scratch_addr[dev] = p;
    }
    scratch = moe::g_scratch_addr[dev];
  }
  // every count the sort reads is written by its histogram kernel first, so
  // the array needs no clearing between calls
  return moe_ragged_sort(topk_ids, T, k, E, x_q, x_scale, D, mode, sorted_src, pos, group_sizes, group_offsets,
                         xs_q, xs_scale, scratch, moe::kNoAllocScratchBytes, stream);
}
