// Row-wise absmax quantisation to e4m3 and the fused producers that feed it:
//   moe_quantize_rows, moe_quantize_weights        (plain bf16 rows)
//   moe_quantize_weights_int8                      (int8 codes, amax / 127)
//   moe_swiglu_quant                               (h = bf16(silu(a0) a1))
//   moe_gather_scale_quant                         (dO = bf16(w G[src]))
//   moe_swiglu_bwd_quant                           (dA0 | dA1)
//   moe_quantize_group_cols                        (per-(expert, column) scales)
//
// All of these are HBM-bound.  One CTA handles one row: each thread loads
// 16-byte vectors (8 bf16; two adjacent ones a unit for most producers),
// applies the producer, keeps the bf16 results in registers, the CTA reduces
// the absolute maximum (warp shuffles, then shared memory; or shuffles among
// the lanes of one 128-column block), and the codes are written with 8- or
// 16-byte stores.  Scales follow "Support quantization for
// tokamax gmm v2" (absmax for activations and gradients) and "Quantize
// activations before EP all gather" (quantise before the sort); weights are
// pre-quantised as in "Keep qwix out of tpu-inference's fused MoE kernel and
// pre-quantize weights" ([E, blocks, 1, N] scales).
#include "common.cuh"

namespace moe {
namespace {

__device__ unsigned int g_err;

constexpr int kThreads = 256;
// Row-kernel mode of the MXFP8 variant (beside the moe_scale_mode values):
// one E8M0 code per row and per 32 columns
constexpr int kModeMx32 = 4;

__device__ __forceinline__ uint4 ldg16(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

__device__ __forceinline__ void unpack8(const uint4& d, float* v) {
  v[0] = bf16lo(d.x);
  v[1] = bf16hi(d.x);
  v[2] = bf16lo(d.y);
  v[3] = bf16hi(d.y);
  v[4] = bf16lo(d.z);
  v[5] = bf16hi(d.z);
  v[6] = bf16lo(d.w);
  v[7] = bf16hi(d.w);
}

__device__ __forceinline__ uint4 pack8(const float* v) {
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}


__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Where the scale of (row, 128-column block b) goes; MXFP8: the E8M0 code of
// (row, 32-column block b) goes to sf[((b / 4) * nrows + row) * 4 + b % 4]
// (K-block-major: the four codes of a row's 128-column block are one word,
// and the words of consecutive rows are adjacent).
struct ScaleOut {
  float* scale;
  int64_t group_n;  // > 0: weights [E, KB, N] with row = e * N + n; 0: [rows, KB]
  int kb;
  uint8_t* sf;
  int64_t nrows;
  __device__ __forceinline__ int64_t blk(int64_t row, int b) const {
    if (group_n > 0) {
      const int64_t e = row / group_n, n = row - e * group_n;
      return (e * kb + b) * group_n + n;
    }
    return row * kb + b;
  }
};

// ---- producers: each "unit" yields U vectors of 8 bf16-exact values ------

struct RowsOp {  // plain bf16 rows
  __device__ __forceinline__ int ndst() const { return 1; }
  __device__ __forceinline__ int64_t dst(int64_t row, int) const { return row; }
  static constexpr int U = 2;
  static constexpr bool kWide = true;
  const uint16_t* x;
  int64_t cols;
  __device__ __forceinline__ void operator()(int64_t row, int u, float (&v)[2][8]) const {
    const uint16_t* r = x + row * cols + 16 * static_cast<int64_t>(u);
    unpack8(ldg16(r), v[0]);
    unpack8(ldg16(r + 8), v[1]);
  }
  __device__ __forceinline__ int64_t col(int u, int uu) const { return 16 * static_cast<int64_t>(u) + 8 * uu; }
};

// h = bf16(silu(a0) * a1), a = [a0 | a1] of width 2F.  WIDE: 16 adjacent
// columns a unit (two vectors); else 8 (measured faster for the per-token h
// scale of long rows, where the row-wide maximum keeps every value in
// registers until the codes are made).
template <bool WIDE>
struct SwigluOpT {
  __device__ __forceinline__ int ndst() const { return 1; }
  __device__ __forceinline__ int64_t dst(int64_t row, int) const { return row; }
  static constexpr int U = WIDE ? 2 : 1;
  static constexpr bool kWide = WIDE;
  const uint16_t* a;
  int64_t F;
  __device__ __forceinline__ void operator()(int64_t row, int u, float (&v)[U][8]) const {
    const uint16_t* r = a + row * 2 * F + 8 * U * static_cast<int64_t>(u);
#pragma unroll
    for (int uu = 0; uu < U; ++uu) {
      float a0[8], a1[8];
      unpack8(ldg16(r + 8 * uu), a0);
      unpack8(ldg16(r + F + 8 * uu), a1);
      uint32_t hb[4];
      swiglu_h_x2<8>(a0, a1, v[uu], hb);
    }
  }
  __device__ __forceinline__ int64_t col(int u, int uu) const { return 8 * U * static_cast<int64_t>(u) + 8 * uu; }
};

struct GatherScaleOp {  // dO[r] = bf16(w[i] * G[i / k]), i = sorted_src[r]; also stores dO
  __device__ __forceinline__ int ndst() const { return 1; }
  __device__ __forceinline__ int64_t dst(int64_t row, int) const { return row; }
  static constexpr int U = 2;
  static constexpr bool kWide = true;
  const uint16_t* G;
  const float* w;
  const int32_t* sorted_src;
  int64_t R;
  int k;
  int64_t D;
  uint16_t* dO;
  __device__ __forceinline__ void operator()(int64_t row, int u, float (&v)[2][8]) const {
    const int64_t i = __ldg(sorted_src + row);
    const int64_t c = 16 * static_cast<int64_t>(u);
    if (i < 0 || i >= R) {
#pragma unroll
      for (int uu = 0; uu < 2; ++uu)
#pragma unroll
        for (int j = 0; j < 8; ++j) v[uu][j] = 0.0f;
    } else {
      const float wi = w ? __ldg(w + i) : 1.0f;
      const uint16_t* src = G + (i / k) * D + c;
      const uint4 d0 = ldg16(src), d1 = ldg16(src + 8);
#pragma unroll
      for (int uu = 0; uu < 2; ++uu) {
        float g[8];
        unpack8(uu ? d1 : d0, g);
#pragma unroll
        for (int j = 0; j < 8; ++j) v[uu][j] = round_bf16(__fmul_rn(wi, g[j]));
      }
    }
    *reinterpret_cast<uint4*>(dO + row * D + c) = pack8(v[0]);
    *reinterpret_cast<uint4*>(dO + row * D + c + 8) = pack8(v[1]);
  }
  __device__ __forceinline__ int64_t col(int u, int uu) const { return 16 * static_cast<int64_t>(u) + 8 * uu; }
};

// plain bf16 token rows whose codes and scales go to the k sorted rows of the
// token (pos[t * k + j]): the quantisation of step 1 fused into the gather of
// step 2 (gather(quantize(x)) == quantize(gather(x)) row by row)
struct RowsGatherOp {
  static constexpr int U = 2;
  static constexpr bool kWide = true;
  const uint16_t* x;
  int64_t cols;
  const int32_t* pos;
  int k;
  int64_t R;
  __device__ __forceinline__ int ndst() const { return k; }
  __device__ __forceinline__ int64_t dst(int64_t row, int j) const {
    const int64_t p = __ldg(pos + row * k + j);
    return (p >= 0 && p < R) ? p : -1;
  }
  __device__ __forceinline__ void operator()(int64_t row, int u, float (&v)[2][8]) const {
    const uint16_t* r = x + row * cols + 16 * static_cast<int64_t>(u);
    unpack8(ldg16(r), v[0]);
    unpack8(ldg16(r + 8), v[1]);
  }
  __device__ __forceinline__ int64_t col(int u, int uu) const { return 16 * static_cast<int64_t>(u) + 8 * uu; }
};

// sigma' chain of the SwiGLU backward, in a fixed order of fp32 operations:
// silu' = sigma (1 + z (1 - sigma)), dA0 = (dH a1) silu', dA1 = dH silu.
__device__ __forceinline__ void bwd_elem(float z, float a1, float dh, float sig, float silu, float& da0, float& da1) {
  const float t1 = __fsub_rn(1.0f, sig);
  const float t2 = __fmul_rn(z, t1);
  const float t3 = __fadd_rn(1.0f, t2);
  const float ds = __fmul_rn(sig, t3);
  const float p = __fmul_rn(dh, a1);
  da0 = round_bf16(__fmul_rn(p, ds));
  da1 = round_bf16(__fmul_rn(dh, silu));
}

struct SwigluBwdOp {  // dA0 = (dH a1) silu'(a0), dA1 = dH silu(a0); also stores dA
  __device__ __forceinline__ int ndst() const { return 1; }
  __device__ __forceinline__ int64_t dst(int64_t row, int) const { return row; }
  static constexpr int U = 2;        // dA0 and dA1 columns (F apart)
  static constexpr bool kWide = false;
  const uint16_t* dH;
  const uint16_t* a;
  int64_t F;
  uint16_t* dA;
  __device__ __forceinline__ void operator()(int64_t row, int u, float (&v)[2][8]) const {
    float z[8], a1[8], dh[8];
    const int64_t c = 8 * static_cast<int64_t>(u);
    unpack8(ldg16(a + row * 2 * F + c), z);
    unpack8(ldg16(a + row * 2 * F + F + c), a1);
    unpack8(ldg16(dH + row * F + c), dh);
    bool fast = true;
#pragma unroll
    for (int j = 0; j < 8; ++j) fast = fast && swiglu_fast_range(z[j]);
    bool ok = fast;
    if (fast) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float d = __fadd_rn(1.0f, exp_fast(-z[j]));
        const float sig = div_checked(1.0f, d, ok);
        const float silu = div_checked(z[j], d, ok);
        bwd_elem(z[j], a1[j], dh[j], sig, silu, v[0][j], v[1][j]);
      }
    }
    if (!ok) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float d = __fadd_rn(1.0f, exp_f32(-z[j]));
        bwd_elem(z[j], a1[j], dh[j], __fdiv_rn(1.0f, d), __fdiv_rn(z[j], d), v[0][j], v[1][j]);
      }
    }
    *reinterpret_cast<uint4*>(dA + row * 2 * F + c) = pack8(v[0]);
    *reinterpret_cast<uint4*>(dA + row * 2 * F + F + c) = pack8(v[1]);
  }
  __device__ __forceinline__ int64_t col(int u, int uu) const { return 8 * static_cast<int64_t>(u) + uu * F; }
};

// ---- the row kernel ------------------------------------------------------
// MODE: MOE_SCALE_PER_ROW, MOE_SCALE_PER_ROW_BLOCK128, MOE_SCALE_PER_TENSOR
// or kModeMx32 (MXFP8, OCP MX v1.0: per 32-column block the shared exponent
// X = floor(log2(amax)) - 8 and codes e4m3(x / 2^X), the division exact).
// MAXI: units per thread (ceil(nunits / blockDim.x) <= MAXI).  I8: int8
// codes instead (int8 weights: scale amax / 127, codes the nearest integers
// of the exact fp32 quotients, ties to even).
template <int MODE, int MAXI, bool I8, class Op>
__global__ void __launch_bounds__(kThreads) rowquant_kernel(Op op, int nunits, int64_t qcols,
                                                            const float* static_scale, uint8_t* q, ScaleOut so) {
  constexpr int U = Op::U;
  static_assert(!Op::kWide || U % 2 == 0, "a wide unit is pairs of adjacent 8-column vectors");
  constexpr int kBlockLanes = Op::kWide ? 8 : 16;  // units per 128-column block
  constexpr int kMxLanes = Op::kWide ? 2 : 4;      // units per 32-column block
  static_assert(MODE != kModeMx32 || Op::kWide, "MXFP8 rows use 16-column units");
  static_assert(!I8 || MODE != kModeMx32, "int8 codes take fp32 scales");
  const int64_t row = blockIdx.x;
  const int tid = threadIdx.x;
  uint32_t pk[MAXI][U][4];
  float amax_i[MAXI];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < MAXI; ++i) {
    const int u = i * blockDim.x + tid;
    float m = 0.0f;
    if (u < nunits) {
      float v[U][8];
      op(row, u, v);
#pragma unroll
      for (int uu = 0; uu < U; ++uu) {
#pragma unroll
        for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[uu][j]));
#pragma unroll
        for (int j = 0; j < 4; ++j) pk[i][uu][j] = pack_bf16x2(v[uu][2 * j], v[uu][2 * j + 1]);
      }
    }
    amax_i[i] = m;
    amax = fmaxf(amax, m);
  }

  float s_row = 1.0f;
  if (MODE == MOE_SCALE_PER_ROW) {
    __shared__ float red[kThreads / 32];
    amax = warp_max(amax);
    if ((tid & 31) == 0) red[tid >> 5] = amax;
    __syncthreads();
    if (tid < 32) {
      float t = tid < static_cast<int>(blockDim.x >> 5) ? red[tid] : 0.0f;
      t = warp_max(t);
      if (tid == 0) red[0] = t;
    }
    __syncthreads();
    s_row = I8 ? int8_scale(red[0]) : absmax_scale(red[0]);
  } else if (MODE == MOE_SCALE_PER_TENSOR) {
    s_row = __ldg(static_scale);
  }

  // codes (and 128-column block scales) once; then written to every destination row
  const float inv_row = __frcp_rn(s_row);
  uint2 codes[MAXI][U];
  float s_blk[MAXI];
  uint8_t e8m0[MAXI];
#pragma unroll
  for (int i = 0; i < MAXI; ++i) {
    const int u = i * blockDim.x + tid;
    float s = s_row, inv = inv_row;
    if (MODE == kModeMx32) {
      // the units of one 32-column block sit on consecutive lanes
      float m = amax_i[i];
#pragma unroll
      for (int o = kMxLanes / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      const int X = mx_shared_exp(m);
      e8m0[i] = static_cast<uint8_t>(X + 127);
      inv = mx_inv_scale(X);
      if (u < nunits) {
#pragma unroll
        for (int uu = 0; uu < U; ++uu) {
          float v[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            v[2 * j] = __fmul_rn(bf16lo(pk[i][uu][j]), inv);  // exact: a power of two
            v[2 * j + 1] = __fmul_rn(bf16hi(pk[i][uu][j]), inv);
          }
          codes[i][uu] = pack_e4m3x8(v);
        }
      }
      continue;
    }
    if (MODE == MOE_SCALE_PER_ROW_BLOCK128) {
      // the units of one 128-column block (16 of 8 columns, or 8 of 16) sit
      // on consecutive lanes
      float m = amax_i[i];
#pragma unroll
      for (int o = kBlockLanes / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      s = I8 ? int8_scale(m) : absmax_scale(m);
      inv = __frcp_rn(s);
    }
    s_blk[i] = s;
    if (u < nunits) {
#pragma unroll
      for (int uu = 0; uu < U; ++uu) {
        float x8[8], v[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          x8[2 * j] = bf16lo(pk[i][uu][j]);
          x8[2 * j + 1] = bf16hi(pk[i][uu][j]);
        }
        if (I8) {  // weights are quantised once, outside the step: the exact quotients
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = __fdiv_rn(x8[j], s);
          codes[i][uu] = pack_i8x8(v);
        } else {
          quant_n<8>(x8, s, inv, v);
          codes[i][uu] = pack_e4m3x8(v);
        }
      }
    }
  }
  for (int d = 0; d < op.ndst(); ++d) {
    const int64_t drow = op.dst(row, d);
    if (drow < 0) continue;
    if (MODE == MOE_SCALE_PER_ROW && tid == 0) so.scale[drow] = s_row;
#pragma unroll
    for (int i = 0; i < MAXI; ++i) {
      const int u = i * blockDim.x + tid;
      if (u < nunits) {
        if (MODE == MOE_SCALE_PER_ROW_BLOCK128 && (u & (kBlockLanes - 1)) == 0)
          so.scale[so.blk(drow, u / kBlockLanes)] = s_blk[i];
        if (MODE == kModeMx32 && (u & (kMxLanes - 1)) == 0) {
          const int b = u / kMxLanes;  // 32-column block
          so.sf[((b >> 2) * so.nrows + drow) * 4 + (b & 3)] = e8m0[i];
        }
        if (Op::kWide) {  // each pair of vectors: 16 adjacent columns, one 16-byte store
#pragma unroll
          for (int uu = 0; uu < U; uu += 2)
            *reinterpret_cast<uint4*>(q + drow * qcols + op.col(u, uu)) =
                make_uint4(codes[i][uu].x, codes[i][uu].y, codes[i][uu + 1].x, codes[i][uu + 1].y);
        } else {
#pragma unroll
          for (int uu = 0; uu < U; ++uu)
            *reinterpret_cast<uint2*>(q + drow * qcols + op.col(u, uu)) = codes[i][uu];
        }
      }
    }
  }
}

template <int MODE, int MAXI, bool I8, class Op>
cudaError_t launch_rows_t(const Op& op, int64_t rows, int nunits, int threads, int64_t qcols, const float* ss,
                          uint8_t* q, ScaleOut so, cudaStream_t st) {
  rowquant_kernel<MODE, MAXI, I8, Op><<<static_cast<unsigned>(rows), threads, 0, st>>>(op, nunits, qcols, ss, q, so);
  return cudaGetLastError();
}

template <int MODE, bool I8, class Op>
cudaError_t launch_rows_m(const Op& op, int64_t rows, int nunits, int64_t qcols, const float* ss, uint8_t* q,
                          ScaleOut so, cudaStream_t st) {
  int threads = nunits >= kThreads ? kThreads : ((nunits + 31) / 32) * 32;
  const int per = (nunits + threads - 1) / threads;
  if (per <= 1) return launch_rows_t<MODE, 1, I8>(op, rows, nunits, threads, qcols, ss, q, so, st);
  if (per <= 2) return launch_rows_t<MODE, 2, I8>(op, rows, nunits, threads, qcols, ss, q, so, st);
  if (per <= 4) return launch_rows_t<MODE, 4, I8>(op, rows, nunits, threads, qcols, ss, q, so, st);
  if (per <= 8) return launch_rows_t<MODE, 8, I8>(op, rows, nunits, threads, qcols, ss, q, so, st);
  return launch_rows_t<MODE, 16, I8>(op, rows, nunits, threads, qcols, ss, q, so, st);
}

template <bool I8 = false, class Op>
moe_status launch_rows(const Op& op, int64_t rows, int nunits, int64_t qcols, moe_scale_mode mode, const float* ss,
                       uint8_t* q, ScaleOut so, cudaStream_t st) {
  if (rows == 0) return MOE_OK;
  cudaError_t e;
  if (mode == MOE_SCALE_PER_ROW)
    e = launch_rows_m<MOE_SCALE_PER_ROW, I8>(op, rows, nunits, qcols, ss, q, so, st);
  else if (mode == MOE_SCALE_PER_ROW_BLOCK128)
    e = launch_rows_m<MOE_SCALE_PER_ROW_BLOCK128, I8>(op, rows, nunits, qcols, ss, q, so, st);
  else
    e = launch_rows_m<MOE_SCALE_PER_TENSOR, I8>(op, rows, nunits, qcols, ss, q, so, st);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

template <class Op>
moe_status launch_rows_mx(const Op& op, int64_t rows, int nunits, int64_t qcols, uint8_t* q, ScaleOut so,
                          cudaStream_t st) {
  if (rows == 0) return MOE_OK;
  return launch_rows_m<kModeMx32, false>(op, rows, nunits, qcols, nullptr, q, so, st) == cudaSuccess ? MOE_OK
                                                                                            : MOE_ERR_CUDA;
}

constexpr int64_t kMaxCols = 16 * kThreads * 8;  // 32768 values per quantised row

moe_status check_mode_ptrs(moe_scale_mode mode, const float* static_scale, const float* scale) {
  if (mode == MOE_SCALE_PER_TENSOR) return static_scale ? MOE_OK : MOE_ERR_INVALID_ARG;
  if (mode == MOE_SCALE_PER_ROW || mode == MOE_SCALE_PER_ROW_BLOCK128)
    return (scale && aligned16(scale)) ? MOE_OK : MOE_ERR_INVALID_ARG;
  return MOE_ERR_INVALID_ARG;
}

// ---- per-(expert, column) gradient quantisation -------------------------
// CTA tile: 256 columns x 256 rows; each warp owns a strip of 32 consecutive
// rows, each lane 8 consecutive columns (one 16-byte load per row).  Rows are
// read 8 at a time (8 loads in flight per thread) and walk through the groups
// in order, so a lane keeps one running maximum per column and flushes it with
// atomicMax (the bit pattern of a non-negative float orders like an unsigned
// integer) only when its strip crosses into the next group.  The scale array
// holds the maxima until a second kernel turns them into amax / 448; a third
// pass quantises against them.
constexpr int kGcRows = 256;
constexpr int kGcStrip = 32;
constexpr int kMaxGroups = 1024;

// Global start row of every group, for groups [0, E]; computed by warp 0.
__device__ __forceinline__ void group_starts_smem(const int32_t* sizes, int E, int64_t* starts) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int64_t carry = 0;
    for (int c = 0; c < E; c += 32) {
      const int g = c + lane;
      int64_t v = g < E ? __ldg(sizes + g) : 0;
      int64_t incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (g < E) starts[g] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) starts[E] = carry;
  }
  __syncthreads();
}

__device__ __forceinline__ int find_group(const int64_t* starts, int E, int64_t m) {
  int lo = 0, hi = E;  // starts[lo] <= m < starts[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (starts[mid] <= m) lo = mid; else hi = mid;
  }
  return lo;
}

template <bool QUANT>
__global__ void __launch_bounds__(256) group_cols_kernel(const uint16_t* g, int64_t M, int64_t N,
                                                         const int32_t* sizes, int E, int g0, int El, uint8_t* q,
                                                         float* scale) {
  __shared__ int64_t starts[kMaxGroups + 1];
  group_starts_smem(sizes, E, starts);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t c0 = (static_cast<int64_t>(blockIdx.x) * 32 + lane) * 8;
  if (c0 >= N) return;
  const int64_t lo = starts[g0], hi = starts[g0 + El];
  int64_t r0 = static_cast<int64_t>(blockIdx.y) * kGcRows + warp * kGcStrip;
  int64_t r1 = min(r0 + kGcStrip, M);
  r0 = max(r0, lo);
  r1 = min(r1, hi);
  if (r0 >= r1) return;
  int grp = find_group(starts, E, r0);  // global group of row r0
  int64_t gend = starts[grp + 1];
  float m[8], sc[8], inv[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) m[j] = 0.0f;
  auto load_scales = [&](int gg) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      sc[j] = scale[static_cast<int64_t>(gg - g0) * N + c0 + j];
      inv[j] = __frcp_rn(sc[j]);
    }
  };
  auto flush = [&](int gg) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      atomicMax(reinterpret_cast<unsigned int*>(scale) + static_cast<int64_t>(gg - g0) * N + c0 + j,
                __float_as_uint(m[j]));
#pragma unroll
    for (int j = 0; j < 8; ++j) m[j] = 0.0f;
  };
  if (QUANT) load_scales(grp);
  for (int64_t rb = r0; rb < r1; rb += 8) {
    uint4 d[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (rb + i < r1) d[i] = __ldg(reinterpret_cast<const uint4*>(g + (rb + i) * N + c0));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t row = rb + i;
      if (row >= r1) break;
      while (row >= gend) {  // next group (rows walk forward through the groups)
        if (!QUANT) flush(grp);
        ++grp;
        gend = starts[grp + 1];
        if (QUANT) load_scales(grp);
      }
      const uint32_t w[4] = {d[i].x, d[i].y, d[i].z, d[i].w};
      float v[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[2 * j] = bf16lo(w[j]);
        v[2 * j + 1] = bf16hi(w[j]);
      }
      if (QUANT) {
        float y[8];
        bool slow = false;
#pragma unroll
        for (int j = 0; j < 8; j += 2) {  // products in pairs (packed fp32, one rounding each)
          f2_unpack(f2_mul(f2_pack(v[j], v[j + 1]), f2_pack(inv[j], inv[j + 1])), y[j], y[j + 1]);
          slow = slow || quant_needs_division(y[j]) || quant_needs_division(y[j + 1]);
        }
        if (slow) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (quant_needs_division(y[j])) y[j] = __fdiv_rn(v[j], sc[j]);
        }
        *reinterpret_cast<uint2*>(q + row * N + c0) = pack_e4m3x8(y);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) m[j] = fmaxf(m[j], fabsf(v[j]));
      }
    }
  }
  if (!QUANT) flush(grp);
}

__global__ void finalize_scales_kernel(float* scale, int64_t n) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) scale[i] = absmax_scale(scale[i]);
}

}  // namespace
}  // namespace moe

using namespace moe;

// Device error word of this translation unit (read by moe_get_device_error).
extern "C" __attribute__((visibility("hidden"))) cudaError_t moe_detail_take_error_quantize(unsigned int* out) {
  unsigned int v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_err, sizeof(v));
  if (e == cudaSuccess && v) e = cudaMemcpyToSymbol(g_err, &z, sizeof(z));
  *out = v;
  return e;
}

// Step 1 fused into the gather of step 2 (moe_quantize_sort): token rows of
// x are quantised once and their codes and scales written to the k sorted
// rows pos[t * k + j]; called by sort.cu once the sort indices exist.
extern "C" __attribute__((visibility("hidden"))) moe_status moe_detail_quantize_gather(
    const uint16_t* x, const int32_t* pos, int64_t T, int k, int64_t D, moe_scale_mode mode, const float* static_scale,
    uint8_t* xs_q, float* xs_scale, cudaStream_t st) {
  MOE_HOST_CHECK(D % 16 == 0 && D <= kMaxCols, MOE_ERR_INVALID_ARG);
  moe_status stt = check_mode_ptrs(mode, static_scale, xs_scale);
  if (stt != MOE_OK) return stt;
  RowsGatherOp op{x, D, pos, k, T * k};
  ScaleOut so{xs_scale, 0, static_cast<int>((D + 127) / 128), nullptr, 0};
  return launch_rows(op, T, static_cast<int>(D / 16), D, mode, static_scale, xs_q, so, st);
}

// MXFP8 form of the fused step 1 + gather (moe_quantize_sort_mx).
extern "C" __attribute__((visibility("hidden"))) moe_status moe_detail_quantize_gather_mx(
    const uint16_t* x, const int32_t* pos, int64_t T, int k, int64_t D, uint8_t* xs_q, uint8_t* xs_sf,
    cudaStream_t st) {
  MOE_HOST_CHECK(D % 128 == 0 && D <= kMaxCols, MOE_ERR_INVALID_ARG);
  RowsGatherOp op{x, D, pos, k, T * k};
  ScaleOut so{nullptr, 0, 0, xs_sf, T * k};
  return launch_rows_mx(op, T, static_cast<int>(D / 16), D, xs_q, so, st);
}

extern "C" moe_status moe_quantize_rows_mx(const uint16_t* x, int64_t rows, int64_t cols, uint8_t* q, uint8_t* sf,
                                           moe_stream_t stream) {
  MOE_HOST_CHECK(x && q && sf && rows >= 0 && cols > 0 && cols % 128 == 0 && cols <= kMaxCols, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(rows < (1ll << 31) && aligned16(x) && aligned16(q), MOE_ERR_INVALID_ARG);
  RowsOp op{x, cols};
  ScaleOut so{nullptr, 0, 0, sf, rows};
  return launch_rows_mx(op, rows, static_cast<int>(cols / 16), cols, q, so, as_stream(stream));
}

extern "C" moe_status moe_swiglu_quant_mx(const uint16_t* a, int64_t R, int64_t F, uint8_t* h_q, uint8_t* h_sf,
                                          moe_stream_t stream) {
  MOE_HOST_CHECK(a && h_q && h_sf && R >= 0 && F > 0 && F % 128 == 0 && F <= kMaxCols, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(R < (1ll << 31) && aligned16(a) && aligned16(h_q), MOE_ERR_INVALID_ARG);
  SwigluOpT<true> op{a, F};
  ScaleOut so{nullptr, 0, 0, h_sf, R};
  return launch_rows_mx(op, R, static_cast<int>(F / 16), F, h_q, so, as_stream(stream));
}

extern "C" moe_status moe_quantize_rows(const uint16_t* x, int64_t rows, int64_t cols, moe_scale_mode mode,
                                        const float* static_scale, uint8_t* q, float* scale, moe_stream_t stream) {
  MOE_HOST_CHECK(x && q && rows >= 0 && cols > 0 && cols % 16 == 0 && cols <= kMaxCols, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(rows < (1ll << 31) && aligned16(x) && aligned16(q), MOE_ERR_INVALID_ARG);
  moe_status st = check_mode_ptrs(mode, static_scale, scale);
  if (st != MOE_OK) return st;
  RowsOp op{x, cols};
  ScaleOut so{scale, 0, static_cast<int>((cols + 127) / 128), nullptr, 0};
  return launch_rows(op, rows, static_cast<int>(cols / 16), cols, mode, static_scale, q, so, as_stream(stream));
}

extern "C" moe_status moe_quantize_weights(const uint16_t* w, int64_t E, int64_t N, int64_t K, moe_scale_mode mode,
                                           const float* static_scale, uint8_t* q, float* scale,
                                           moe_stream_t stream) {
  MOE_HOST_CHECK(w && q && E > 0 && N > 0 && K > 0 && K % 16 == 0 && K <= kMaxCols, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(E * N < (1ll << 31) && aligned16(w) && aligned16(q), MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(mode != MOE_SCALE_PER_ROW_BLOCK128 || K % 128 == 0, MOE_ERR_INVALID_ARG);
  moe_status st = check_mode_ptrs(mode, static_scale, scale);
  if (st != MOE_OK) return st;
  RowsOp op{w, K};
  ScaleOut so{scale, N, static_cast<int>(K / 128), nullptr, 0};
  return launch_rows(op, E * N, static_cast<int>(K / 16), K, mode, static_scale, q, so, as_stream(stream));
}

extern "C" moe_status moe_quantize_weights_int8(const uint16_t* w, int64_t E, int64_t N, int64_t K,
                                                moe_scale_mode mode, const float* static_scale, int8_t* q,
                                                float* scale, moe_stream_t stream) {
  MOE_HOST_CHECK(w && q && E > 0 && N > 0 && K > 0 && K % 16 == 0 && K <= kMaxCols, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(E * N < (1ll << 31) && aligned16(w) && aligned16(q), MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(mode != MOE_SCALE_PER_ROW_BLOCK128 || K % 128 == 0, MOE_ERR_INVALID_ARG);
  moe_status st = check_mode_ptrs(mode, static_scale, scale);
  if (st != MOE_OK) return st;
  RowsOp op{w, K};
  ScaleOut so{scale, N, static_cast<int>(K / 128), nullptr, 0};
  return launch_rows<true>(op, E * N, static_cast<int>(K / 16), K, mode, static_scale, reinterpret_cast<uint8_t*>(q),
                           so, as_stream(stream));
}

extern "C" moe_status moe_swiglu_quant(const uint16_t* a, int64_t R, int64_t F, moe_scale_mode mode,
                                       const float* static_scale, uint8_t* h_q, float* h_scale,
                                       moe_stream_t stream) {
  MOE_HOST_CHECK(a && h_q && R >= 0 && F > 0 && F % 16 == 0 && F <= kMaxCols, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(R < (1ll << 31) && aligned16(a) && aligned16(h_q), MOE_ERR_INVALID_ARG);
  moe_status st = check_mode_ptrs(mode, static_scale, h_scale);
  if (st != MOE_OK) return st;
  ScaleOut so{h_scale, 0, static_cast<int>((F + 127) / 128), nullptr, 0};
  if (mode == MOE_SCALE_PER_ROW) {
    SwigluOpT<false> op{a, F};
    return launch_rows(op, R, static_cast<int>(F / 8), F, mode, static_scale, h_q, so, as_stream(stream));
  }
  SwigluOpT<true> op{a, F};
  return launch_rows(op, R, static_cast<int>(F / 16), F, mode, static_scale, h_q, so, as_stream(stream));
}

extern "C" moe_status moe_gather_scale_quant(const uint16_t* G, const float* w, const int32_t* sorted_src,
                                             int64_t T, int k, int64_t D, uint16_t* dO, uint8_t* dO_q,
                                             float* dO_scale, moe_stream_t stream) {
  MOE_HOST_CHECK(G && sorted_src && dO && dO_q && dO_scale && T >= 0 && k > 0 && D > 0, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(D % 16 == 0 && D <= kMaxCols && T <= ((1ll << 31) - 1) / k, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(aligned16(G) && aligned16(dO) && aligned16(dO_q) && aligned16(dO_scale), MOE_ERR_INVALID_ARG);
  GatherScaleOp op{G, w, sorted_src, T * k, k, D, dO};
  ScaleOut so{dO_scale, 0, 0, nullptr, 0};
  return launch_rows(op, T * k, static_cast<int>(D / 16), D, MOE_SCALE_PER_ROW, nullptr, dO_q, so,
                     as_stream(stream));
}

extern "C" moe_status moe_swiglu_bwd_quant(const uint16_t* dH, const uint16_t* a, int64_t R, int64_t F,
                                           uint16_t* dA, uint8_t* dA_q, float* dA_scale, moe_stream_t stream) {
  MOE_HOST_CHECK(dH && a && dA && dA_q && dA_scale && R >= 0 && F > 0, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(F % 16 == 0 && 2 * F <= kMaxCols && R < (1ll << 31), MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(aligned16(dH) && aligned16(a) && aligned16(dA) && aligned16(dA_q) && aligned16(dA_scale),
                 MOE_ERR_INVALID_ARG);
  SwigluBwdOp op{dH, a, F, dA};
  ScaleOut so{dA_scale, 0, 0, nullptr, 0};
  return launch_rows(op, R, static_cast<int>(F / 8), 2 * F, MOE_SCALE_PER_ROW, nullptr, dA_q, so,
                     as_stream(stream));
}

extern "C" moe_status moe_quantize_group_cols(const uint16_t* g, int64_t M, int64_t N, const int32_t* group_sizes,
                                              int E, int group_offset, int E_local, uint8_t* q, float* scale,
                                              moe_stream_t stream) {
  MOE_HOST_CHECK(g && group_sizes && scale && M >= 0 && N > 0 && N % 16 == 0, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(E > 0 && E <= kMaxGroups && group_offset >= 0 && E_local > 0 && group_offset + E_local <= E,
                 MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(aligned16(g) && (q == nullptr || aligned16(q)) && aligned16(scale), MOE_ERR_INVALID_ARG);
  cudaStream_t st = as_stream(stream);
  const int64_t ns = static_cast<int64_t>(E_local) * N;
  MOE_CUDA_TRY(cudaMemsetAsync(scale, 0, sizeof(float) * ns, st));
  if (M > 0) {
    dim3 grid(static_cast<unsigned>((N / 8 + 31) / 32), static_cast<unsigned>((M + kGcRows - 1) / kGcRows));
    group_cols_kernel<false><<<grid, 256, 0, st>>>(g, M, N, group_sizes, E, group_offset, E_local, q, scale);
    MOE_CUDA_TRY(cudaGetLastError());
  }
  finalize_scales_kernel<<<static_cast<unsigned>((ns + 255) / 256), 256, 0, st>>>(scale, ns);
  MOE_CUDA_TRY(cudaGetLastError());
  if (M > 0 && q != nullptr) {  // q == NULL: the scales only (tgmm_fp8_gcq makes the codes)
    dim3 grid(static_cast<unsigned>((N / 8 + 31) / 32), static_cast<unsigned>((M + kGcRows - 1) / kGcRows));
    group_cols_kernel<true><<<grid, 256, 0, st>>>(g, M, N, group_sizes, E, group_offset, E_local, q, scale);
    MOE_CUDA_TRY(cudaGetLastError());
  }
  return MOE_OK;
}
