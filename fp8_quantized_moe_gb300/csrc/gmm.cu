// Grouped FP8 matmuls on the 5th-generation tensor cores (tcgen05, sm_103a):
//   gmm_fp8   out[m, n] = sum_k deq(lhs)[m, k] deq(rhs)[g(m), n, k]   (bf16 out)
//   tgmm_fp8  out[e, k, n] = sum_{m in e} deq(lhs)[m, k] deq(rhs)[m, n] (fp32 out)
// following "Quantize activations before EP all gather" (gmm_v2 on
// pre-quantised lhs with rhs_scale and group_offset, lhs scale on the
// output, bf16 output), "Support quantization for tokamax gmm v2" (gmm and
// tgmm with absmax scales) and "Keep qwix out of tpu-inference's fused MoE
// kernel and pre-quantize weights" (fp8 weights with [E, blocks, 1, N]
// scales; 32-bit accumulation);
//   gmm_fp8_w8 the same gmm with int8 weights (that page's other weight
//              type), on the f16 MMA (both code types are exact in f16);
// and, not from those pages,
//   gmm_fp8_mx the same gmm on MXFP8 operands (OCP Microscaling Formats v1.0:
//              one E8M0 power-of-two scale per 32 values of K).
//
// Design (one persistent CTA per SM, 1 CTA/SM by shared memory):
//   warp 0      TMA producer: 128x128 A tile + 256x128 B tile per stage into a
//               4-stage ring of 48 KB stages (128-byte swizzle).
//   warp 1      MMA issuer: 4 x tcgen05.mma kind::f8f6f4 (M=128, N=256, K=32)
//               per stage into a TMEM accumulator; commits free the stage.
//               Also allocates / frees the 512 TMEM columns (2 accumulators).
//   warps 2..   epilogue: tcgen05.ld the accumulator, apply the scales, store.
// Accumulators are double-buffered, so the epilogue of tile i overlaps the
// mainloop of tile i+1.  With a blockwise (128-wide K block) scale on either
// operand the scale cannot leave the sum, so every K block gets a fresh TMEM
// accumulator and eight epilogue warps fold it into fp32 registers
// ("promotion", packed f32x2 FMAs).
//
// MXFP8 (gmm_fp8_mx, gmm_fp8_mx_swiglu): tcgen05.mma.kind::mxf8f6f4 with
// one E8M0 scale per 32 values of K on each operand, applied by the tensor
// core, so one accumulator runs over the whole K loop.  A control warp
// gathers each stage's scale codes into shared-memory atoms (a ring of its
// own), and the MMA issuer copies them into tensor memory (tcgen05.cp) ahead
// of the stage's MMAs; the scales' tensor-memory slots take the columns next
// to the accumulator, so there is one accumulator, not two.
//
// Tile scheduler: tiles are ordered expert-major, then N tile, then M tile,
// so that the CTAs running at the same time share the same expert's weights
// (weights stream from HBM about once).  A group's M tiles start at its first
// row; rows past the group end are computed and masked at the store.  tgmm
// contracts over a group's rows: its operands are first transposed into the
// workspace with every group padded (with zeros) to a multiple of 128 rows, so
// that the contraction dimension is contiguous (K-major) and every TMA box
// starts 16-byte aligned.
//
// Every wait is bounded (mbarrier try_wait + %globaltimer); on expiry the
// kernel raises MOE_DEVERR_TIMEOUT, drains what it issued and returns.
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <type_traits>

#include "common.cuh"

namespace moe {
namespace {

__device__ unsigned int g_err;

constexpr int BM = 128;
constexpr int BK = 128;
#ifndef MOE_GMM_NSTAGE
#define MOE_GMM_NSTAGE 4
#endif
constexpr int A_BYTES = BM * BK;
constexpr int UMMA_K = 32;
constexpr int kMaxStages = 8;
constexpr int kMaxAcc = 8;
constexpr int kMaxGroups = 1024;
constexpr int64_t kPairMinK = 3072;  // gmm K from which the plain and SwiGLU gmm run on CTA pairs
constexpr int kMaxDevices = 256;     // host-side per-device caches

enum Mode {
  kFinal = 0,
  kPromote = 1,
  kTgmm = 2,
  kSwiglu = 3,
  kSplit = 4,
  kPromoteSwiglu = 5,
  kBf16 = 6,
  kRouter = 7,
  kMx = 8,         // MXFP8 operands: block-scaled MMAs, bf16 out
  kMxSwiglu = 9    // MXFP8 wi gmm with the SwiGLU and MXFP8 requantisation epilogue
};
constexpr int kStg8Pitch = 80;                  // warp_store_32x32_bf16: staging row pitch (bytes)
constexpr int kStg8Bytes = 8 * kStg8Pitch;      // and its 8-row buffer per warp
constexpr int kMxSfStageBytes = 3 * 512;  // MXFP8: per stage, one A and two B scale-factor atoms (32 x 16 B each)
// MXFP8: slots of the shared-memory scale-factor ring (more than the operand
// stages, so that the gatherer keeps several stages of copies in flight
// without holding back the MMAs)
constexpr int kMxSfSlots = 8;
#ifndef MOE_MX_LAG
#define MOE_MX_LAG 3
#endif
constexpr int kSwSlots = 8;  // promotion: ring of per-K-block weight-scale rows in shared memory

struct Params {
  const int32_t* group_sizes;
  int E, g0, El;
  int64_t M;
  int K, N;
  int kblocks;  // gmm: K blocks per tile
  int kb_split;  // kSplit: K blocks of the first scale segment
  int ntiles;   // N tiles
  int ktiles;   // tgmm: output-row tiles (K / 128)
  const float* lhs_scale;
  int lhs_mode;
  const float* rhs_scale;
  int rhs_mode;
  void* out;
  // kSwiglu: h = bf16(silu(a0) a1) requantised; a = [a0 | a1] optionally kept
  int F;
  int h_mode;
  const float* h_static;
  uint16_t* a_out;     // [M, 2F] bf16 or null
  uint16_t* h_out;     // [M, F] bf16 (per-row h scales)
  uint8_t* h_q;        // [M, F] e4m3 (per-tensor / per-128 h scales)
  float* h_scale;      // per-row: running amax [M]; per-128: [M, F/128]
  // kBf16: fp32 output rows instead of bf16
  int out_f32;
  // test hook: the epilogue first waits (bounded by stall_ns) on a barrier
  // that nothing arrives on, so the bounded-wait timeout path runs
  int stall;
  uint64_t stall_ns;
  // kRouter: softmax top-k of the first `E` logit columns of each row
  int rE, rk;
  float* logits;       // [M, rE] fp32
  int32_t* topk_ids;   // [M, rk]
  float* topk_w;       // [M, rk]
  // MXFP8: E8M0 codes, one per 32 values along K, K-block-major: the four
  // codes of row r's 128-wide K block kb form the word [kb][r] (lhs [K/128]
  // [M], rhs [K/128][E_local * N]); kMxSwiglu also writes h's codes
  // ([F/128][M])
  const uint8_t* lhs_sf;
  const uint8_t* rhs_sf;
  uint8_t* h_sf;
};

struct SmemCtl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[kMaxAcc];
  uint64_t tempty[kMaxAcc];
  uint64_t sffull[kMxSfSlots];   // MXFP8: the slot's scale-factor atoms are in shared memory
  uint64_t sfempty[kMxSfSlots];  // MXFP8: the tensor core has copied the slot out (its MMAs completed)
  uint64_t sfull[kSwSlots];   // promotion: a weight-scale row of the ring has landed
  uint64_t sempty[kSwSlots];  // promotion: a weight-scale row of the ring has been read by every epilogue warp
  uint64_t xbar[4][2];        // promotion + SwiGLU: the two warps of a lane quarter have posted their h maxima
  uint64_t drain;
  uint64_t never;  // test hook: a barrier that nothing arrives on
  uint32_t tmem_base;
  int abort_flag;
  int no_abort;  // always 0: for waits that must run to completion or to their time limit
  int err;
  int total_tiles;
  int gstart[kMaxGroups + 1];       // gmm: first row of local group; tgmm: padded first row
  int tile_prefix[kMaxGroups + 1];  // gmm: first tile of local group
  int gsize[kMaxGroups];
  // per-mode scratch (one mode per kernel)
  alignas(16) float pamax[2][4][4][32];  // fused SwiGLU, per-128 h scales: row maxima of the column parts
};
static_assert(offsetof(SmemCtl, pamax) % 16 == 0, "SmemCtl alignment");
static_assert(sizeof(SmemCtl) % 16 == 0, "SmemCtl size");

// Tile configuration per mode.  The plain and SwiGLU gmm run on CTA pairs (a
// 2-CTA cluster) from K = 3072: one 256x256 MMA per K step over both CTAs,
// each CTA holding 128 rows of A and half of the B tile, so a stage is 32 KB
// per CTA instead of 48 and the operand traffic through each SM's shared
// memory drops by a third.  Promotion (a blockwise operand scale) uses one
// CTA and 128x256 tiles: an M=128 tcgen05 MMA costs about the same time at
// N=128 as at N=256 (measured), so only N=256 keeps the tensor pipe at full
// rate; its two 256-column TMEM accumulators take alternate K blocks, and a
// one-CTA tile keeps the per-block accumulator hand-off local and wastes at
// most 127 rows at the end of a group.  tgmm uses 128x256 tiles with two
// accumulators.
#ifndef MOE_PROMOTE_EPI_WARPS
#define MOE_PROMOTE_EPI_WARPS 8
#endif
#ifndef MOE_PROMOTE_CHUNK
#define MOE_PROMOTE_CHUNK 32
#endif
#ifndef MOE_TGMM_EPI_WARPS
#define MOE_TGMM_EPI_WARPS 8
#endif
#ifndef MOE_TGMM_NSTAGE
#define MOE_TGMM_NSTAGE 3
#endif
#ifndef MOE_TGMM_STG_BUFS
#define MOE_TGMM_STG_BUFS 2
#endif
#ifndef MOE_GMM_PAIR
#define MOE_GMM_PAIR 1
#endif
#ifndef MOE_PAIR_TMEM_COLS
#define MOE_PAIR_TMEM_COLS 512
#endif
template <int MODE, bool PAIR_REQ = false>
struct Cfg {
  static constexpr bool PROMOTE = MODE == kPromote || MODE == kPromoteSwiglu;
  // MXFP8: block-scaled MMAs whose E8M0 scales are copied into tensor memory
  // next to a single accumulator
  static constexpr bool MX = MODE == kMx || MODE == kMxSwiglu;
  // the control warpgroup hands registers to the epilogue (setmaxnreg)
  static constexpr bool SPLIT = PROMOTE || MX;
  static constexpr bool PAIR = PAIR_REQ && MOE_GMM_PAIR && (MODE == kFinal || MODE == kSwiglu);
  // bf16 operands (kind::f16): a 128-byte K block is 64 elements
  static constexpr bool BF = MODE == kBf16 || MODE == kRouter;
  static constexpr int KSTEP = BF ? 64 : 128;  // elements of K per 128-byte block
  static constexpr int BN = 256;  // output columns per tile
  static constexpr int TMEM_COLS = PAIR ? MOE_PAIR_TMEM_COLS : 512;
  static constexpr int SEGS = MODE == kSplit ? 2 : 1;        // accumulators per tile (one per K segment)
  // tiles (promotion: K blocks) in flight in tensor memory; MXFP8 keeps one
  // 256-column accumulator and puts a scale-factor slot per stage after it
  static constexpr int NACC = MX ? 1 : TMEM_COLS / (BN * SEGS);
  static constexpr int SF_COL0 = BN;  // MXFP8: tensor-memory column of stage 0's scale slot (16 columns a stage)
  static constexpr int NSTAGE = PAIR ? 6 : (MODE == kTgmm ? MOE_TGMM_NSTAGE : MOE_GMM_NSTAGE);
  static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * BK;  // this CTA's part of the B tile
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t TX_BYTES = (PAIR ? 2 : 1) * STAGE_BYTES;  // what one full barrier waits for
  static constexpr uint32_t IDESC = BF ? idesc_bf16_f32(BM, BN) : idesc_e4m3_f32(PAIR ? 2 * BM : BM, BN);
  static constexpr int EPI_WARPS =
      PROMOTE ? MOE_PROMOTE_EPI_WARPS : ((MODE == kSwiglu || MX) ? 8 : (MODE == kTgmm ? MOE_TGMM_EPI_WARPS : 4));
  // warps before the epilogue: producer, MMA issuer and, with the register
  // split, two more that complete the control warpgroup (MXFP8: the first of
  // them gathers the scale factors; promotion: both idle)
  static constexpr int CTRL_WARPS = SPLIT ? 4 : 2;
  static constexpr int THREADS = 32 * (CTRL_WARPS + EPI_WARPS);
  // promotion register split: the control warpgroup gives registers to the
  // epilogue warpgroups, whose running sums (256 / (EPI_WARPS / 4) per
  // thread) need them
  static constexpr int LAUNCH_REGS = (65536 / THREADS) & ~7;  // what a thread is launched with at most
  static constexpr uint32_t CTRL_REGS = EPI_WARPS == 8 ? 40 : 32;
  static constexpr uint32_t EPI_REGS = ((LAUNCH_REGS * THREADS - 128 * CTRL_REGS) / (32 * EPI_WARPS)) & ~7u;
  // per-warp staging of 32x32 output blocks: kFinal, bf16 rows padded to 80
  // bytes for row-contiguous stores; kTgmm, two 4 KB fp32 blocks in the
  // 128-byte-swizzled layout of a TMA store box
  static constexpr int STG_PITCH = (MODE == kFinal || MODE == kSplit || MODE == kBf16) ? 80 : 0;
  static constexpr int STG_BUFS = MODE == kTgmm ? MOE_TGMM_STG_BUFS : 1;
  // kSwiglu, kMx, kMxSwiglu: an 8-row staging buffer per warp (warp_store_32x64B)
  static constexpr int STG_WARP_BYTES = (MODE == kFinal || MODE == kSplit || MODE == kBf16)
                                            ? 32 * STG_PITCH
                                            : (MODE == kTgmm ? STG_BUFS * 4096
                                                              : ((MX || MODE == kSwiglu) ? kStg8Bytes : 0));
  static constexpr size_t CTL_BYTES = (sizeof(SmemCtl) + 1023) / 1024 * 1024;  // keeps the staging 1 KB aligned
  // promotion: kSwSlots rows of BN weight scales, one per K block in flight
  static constexpr int SW_RING_BYTES = PROMOTE ? kSwSlots * BN * 4 : 0;
  // MXFP8: each stage's scale-factor atoms
  static constexpr int SF_RING_BYTES = MX ? kMxSfSlots * kMxSfStageBytes : 0;
  static constexpr size_t SMEM = 1024 + static_cast<size_t>(NSTAGE) * STAGE_BYTES + CTL_BYTES +
                                 static_cast<size_t>(EPI_WARPS) * STG_WARP_BYTES + SW_RING_BYTES + SF_RING_BYTES;
  static_assert(NSTAGE <= kMaxStages && NACC >= 1 && NACC <= kMaxAcc && NACC * BN * SEGS <= TMEM_COLS &&
                    STAGE_BYTES % 1024 == 0 && BN % 32 == 0,
                "tile configuration");
  // the producer runs at most NSTAGE K blocks ahead of the MMA, which runs at
  // most NACC ahead of the epilogue: every block in flight has its scale row
  static_assert(!PROMOTE || kSwSlots >= NSTAGE + NACC, "promotion: weight-scale ring too short");
  static_assert(!PROMOTE || EPI_WARPS == 8 || EPI_WARPS == 16, "promotion epilogue: 8 or 16 warps");
  // the split must fit in what the CTA is launched with (the host also
  // checks the kernel's actual register count before the launch)
  static_assert(!SPLIT || (128 * CTRL_REGS + 32 * EPI_WARPS * EPI_REGS <= LAUNCH_REGS * THREADS &&
                           EPI_REGS <= 255 && EPI_REGS >= 96),
                "register split");
  static_assert(!MX || (!PAIR && EPI_WARPS == 8 && SF_COL0 + 16 * NSTAGE <= TMEM_COLS), "MXFP8 configuration");
  static_assert(SMEM <= 232448, "shared memory per CTA");
};

// ---- coalesced row-segment stores ------------------------------------------
// A warp's 32 rows x 64 bytes (32 bf16 columns, or 64 e4m3 codes) to global
// memory: lane r holds row r's 64 bytes in w.  The rows go out 8 at a time
// through an 8-row staging buffer (pitch 80 bytes), each store instruction
// writing 8 rows x 64 contiguous bytes (lane 4 i + q: row i, bytes 16 q ..),
// so that every sector is written whole rather than half by each of 32 rows.
// out points at row 0 and the first byte; rows >= nrows and 16-byte chunks at
// or past nbytes (a multiple of 16 when positive) are skipped.  Every lane of
// the warp calls it.
__device__ __forceinline__ void warp_store_32x64B(uint8_t* stg, const uint32_t (&w)[16], uint8_t* out,
                                                  int64_t pitch, int nrows, int nbytes) {
  const int lane = threadIdx.x & 31;
  const int rr = lane >> 2, q = lane & 3;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    if ((lane >> 3) == s) {
      uint4* d = reinterpret_cast<uint4*>(stg + (lane & 7) * kStg8Pitch);
      d[0] = make_uint4(w[0], w[1], w[2], w[3]);
      d[1] = make_uint4(w[4], w[5], w[6], w[7]);
      d[2] = make_uint4(w[8], w[9], w[10], w[11]);
      d[3] = make_uint4(w[12], w[13], w[14], w[15]);
    }
    __syncwarp();
    const int row = 8 * s + rr;
    if (row < nrows && 16 * q < nbytes)
      *reinterpret_cast<uint4*>(out + row * pitch + 16 * q) =
          *reinterpret_cast<const uint4*>(stg + rr * kStg8Pitch + 16 * q);
    __syncwarp();
  }
}

// ---- group tables --------------------------------------------------------
// Warp 0 reads all E sizes at once (<= 32 per lane), scans them, and fills
// the tables for the local groups [g0, g0 + El).  Returns (in ctl->err) 1 if a
// size is negative or the sizes do not add up to M.  With PAIR a unit of work
// is a pair of M tiles (one per CTA of the pair).
template <bool TGMM, bool PAIR, class Ctl>
__device__ void build_group_tables(const Params& p, Ctl* ctl) {
  const int lane = threadIdx.x & 31;
  int v[kMaxGroups / 32];
#pragma unroll
  for (int c = 0; c < kMaxGroups / 32; ++c) {
    const int g = c * 32 + lane;
    // no size table: one group of all M rows (the router's dense contractions)
    v[c] = g < p.E ? (p.group_sizes ? __ldg(p.group_sizes + g) : static_cast<int>(p.M)) : 0;
  }
  int64_t carry_rows = 0;
  int carry_aux = 0;
  bool bad = false;
#pragma unroll
  for (int c = 0; c < kMaxGroups / 32; ++c) {
    if (c * 32 >= p.E) break;
    const int g = c * 32 + lane;
    const int sz = v[c];
    if (sz < 0) bad = true;
    const int local = g - p.g0;
    const bool mine = g < p.E && local >= 0 && local < p.El;
    int64_t incl = sz;
    // aux: gmm -> tiles of the group; tgmm -> padded rows of the group
    int aux = 0;
    if (mine && sz > 0)
      aux = TGMM ? ((sz + BM - 1) / BM) * BM
                 : (PAIR ? (sz + 2 * BM - 1) / (2 * BM) : (sz + BM - 1) / BM) * p.ntiles;
    int incl_aux = aux;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t t = __shfl_up_sync(0xffffffffu, incl, o);
      const int ta = __shfl_up_sync(0xffffffffu, incl_aux, o);
      if (lane >= o) {
        incl += t;
        incl_aux += ta;
      }
    }
    if (mine) {
      ctl->gsize[local] = sz;
      if (TGMM) {
        ctl->gstart[local] = carry_aux + incl_aux - aux;  // padded start
      } else {
        ctl->gstart[local] = static_cast<int>(carry_rows + incl - sz);
        ctl->tile_prefix[local] = carry_aux + incl_aux - aux;
      }
    }
    carry_rows += __shfl_sync(0xffffffffu, incl, 31);
    carry_aux += __shfl_sync(0xffffffffu, incl_aux, 31);
  }
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) {
    if (TGMM) {
      ctl->gstart[p.El] = carry_aux;
      ctl->total_tiles = p.El * p.ktiles * p.ntiles;
    } else {
      ctl->tile_prefix[p.El] = carry_aux;
      ctl->total_tiles = carry_aux;
    }
    ctl->err = (bad || carry_rows != p.M) ? 1 : 0;
  }
}

struct Tile {
  int el;       // local group
  int nkb;      // K blocks to accumulate (0: empty tgmm group)
  int ax, ay;   // A box coordinates of K block 0 (x advances by BK per block)
  int bx, by;   // B box coordinates of K block 0
  int row0;     // gmm: first output row; tgmm: first output row (k) of the tile
  int rows;     // valid output rows in the tile
  int n0;       // first output column
};

template <int MODE, bool PAIR, class Ctl>
__device__ __forceinline__ Tile get_tile(const Params& p, const Ctl* ctl, int t, int rank) {
  Tile tl;
  constexpr int BN = Cfg<MODE, PAIR>::BN;
  if (MODE == kTgmm) {
    const int per = p.ktiles * p.ntiles;
    tl.el = t / per;
    const int r = t - tl.el * per;
    const int kt = r / p.ntiles, nt = r - kt * p.ntiles;
    const int sz = ctl->gsize[tl.el];
    const int pst = ctl->gstart[tl.el];
    tl.nkb = (sz + BK - 1) / BK;
    tl.ax = pst;
    tl.ay = kt * BM;
    tl.bx = pst;
    tl.by = nt * BN;
    tl.row0 = kt * BM;
    tl.rows = min(BM, p.K - kt * BM);
    tl.n0 = nt * BN;
  } else {
    int lo = 0, hi = p.El;  // tile_prefix[lo] <= t < tile_prefix[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (ctl->tile_prefix[mid] <= t) lo = mid; else hi = mid;
    }
    // skip empty groups that share the same prefix value
    while (lo + 1 < p.El && ctl->tile_prefix[lo + 1] <= t) ++lo;
    tl.el = lo;
    const int sz = ctl->gsize[lo];
    // M tiles of the group, counted in units (pairs of tiles for a CTA pair)
    const int mt = PAIR ? (sz + 2 * BM - 1) / (2 * BM) : (sz + BM - 1) / BM;
    const int local = t - ctl->tile_prefix[lo];
    const int nt = local / mt;
    const int mi = PAIR ? 2 * (local - nt * mt) + rank : local - nt * mt;
    tl.nkb = p.kblocks;
    tl.row0 = ctl->gstart[lo] + mi * BM;
    tl.rows = min(BM, sz - mi * BM);  // <= 0: the odd CTA of a pair past the group's end
    tl.ax = 0;
    tl.ay = tl.row0;
    tl.bx = 0;
    if (MODE == kSwiglu || MODE == kPromoteSwiglu || MODE == kMxSwiglu) {
      // 128 h columns: wi_0 channels nt*128.. and the matching wi_1 channels
      // (a CTA pair: the even CTA holds the wi_0 rows, the odd one the wi_1 rows)
      tl.by = lo * 2 * p.F + nt * 128 + (PAIR ? rank * p.F : 0);
      tl.n0 = nt * 128;
    } else {
      tl.by = lo * p.N + nt * BN + (PAIR ? rank * (BN / 2) : 0);
      tl.n0 = nt * BN;
    }
  }
  return tl;
}

__device__ __forceinline__ float lhs_scale_at(const Params& p, int64_t row, int kb) {
  if (p.lhs_mode == MOE_SCALE_PER_ROW) return __ldg(p.lhs_scale + row);
  if (p.lhs_mode == MOE_SCALE_PER_ROW_BLOCK128) return __ldg(p.lhs_scale + row * p.kblocks + kb);
  return __ldg(p.lhs_scale);
}

// tgmm operand scale: per tensor or per (local group, column).
__device__ __forceinline__ float group_col_scale(const float* s, int mode, int el, int c, int C) {
  return mode == MOE_SCALE_PER_GROUP_COL ? __ldg(s + static_cast<int64_t>(el) * C + c) : __ldg(s);
}

// 32 per-column scales starting at column nb: 16-byte loads from `base` when
// the span is in range and per-column, else guarded scalar loads or the one
// per-tensor value.
__device__ __forceinline__ void load_col_scales32(const float* base, int nb, int N, bool per_col, float uniform,
                                                  float* sw) {
  if (per_col && nb + 32 <= N) {
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const float4 t = __ldg(reinterpret_cast<const float4*>(base + nb) + g);
      sw[4 * g] = t.x;
      sw[4 * g + 1] = t.y;
      sw[4 * g + 2] = t.z;
      sw[4 * g + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) sw[j] = per_col ? (nb + j < N ? __ldg(base + nb + j) : 0.f) : uniform;
  }
}

// The producer's and the MMA issuer's pipeline waits.  Beside the promotion
// epilogue (the bound there) they poll with a suspend-time hint, so that they
// leave issue slots to the epilogue warps of their SM sub-partitions
// (measured 1-2 % faster); elsewhere they poll without one.
#define CTRL_WAIT(...) (C::PROMOTE ? mbar_wait_bounded_idle(__VA_ARGS__) : mbar_wait_bounded(__VA_ARGS__))

template <int MODE, bool PAIR_REQ>
__global__ void __launch_bounds__(Cfg<MODE, PAIR_REQ>::THREADS, 1)
    mma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmO, const Params p) {
  using C = Cfg<MODE, PAIR_REQ>;
  constexpr int EPI_WARPS = C::EPI_WARPS, BN = C::BN, NSTAGE = C::NSTAGE, NACC = C::NACC;
  constexpr int STAGE_BYTES = C::STAGE_BYTES;
  constexpr uint32_t IDESC = C::IDESC;
  constexpr bool PAIR = C::PAIR;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(base_ptr + NSTAGE * STAGE_BYTES);
  uint8_t* stg_base = base_ptr + NSTAGE * STAGE_BYTES + C::CTL_BYTES;  // output staging (kFinal, kTgmm)
  // promotion: ring of per-K-block weight-scale rows (BN floats each)
  float* sw_ring = reinterpret_cast<float*>(stg_base + EPI_WARPS * C::STG_WARP_BYTES);
  // MXFP8: per stage, the A scale atom (rows 32 c + l of the tile in row l,
  // 16 bytes: the E8M0 codes of the stage's four K blocks for c = 0..3) and
  // the two B atoms (tile rows 0..127, 128..255) laid out the same way
  const uint32_t sf_ring = smem_u32(reinterpret_cast<uint8_t*>(sw_ring) + C::SW_RING_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // A CTA pair works on the same sequence of units; its even CTA (rank 0)
  // issues the MMAs and owns the full and accumulator-empty barriers.
  const int rank = PAIR ? static_cast<int>(__clusterRelativeBlockRank()) : 0;
  const int unit0 = PAIR ? static_cast<int>(__clusterIdx().x) : static_cast<int>(blockIdx.x);
  const int units = PAIR ? static_cast<int>(__clusterGridDimInClusters().x) : static_cast<int>(gridDim.x);

  if (warp == 0) build_group_tables<MODE == kTgmm, PAIR>(p, ctl);
  if (threadIdx.x == 32) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int a = 0; a < NACC; ++a) {
      mbar_init(smem_u32(&ctl->tfull[a]), 1);
      mbar_init(smem_u32(&ctl->tempty[a]), (PAIR ? 2 : 1) * EPI_WARPS);
    }
    if (C::MX)
      for (int q = 0; q < kMxSfSlots; ++q) {
        mbar_init(smem_u32(&ctl->sffull[q]), 32);
        mbar_init(smem_u32(&ctl->sfempty[q]), 1);
      }
    if (C::PROMOTE) {
      for (int q = 0; q < kSwSlots; ++q) {
        mbar_init(smem_u32(&ctl->sfull[q]), 1);
        mbar_init(smem_u32(&ctl->sempty[q]), EPI_WARPS);
      }
      for (int q = 0; q < 4; ++q)
        for (int b = 0; b < 2; ++b) mbar_init(smem_u32(&ctl->xbar[q][b]), EPI_WARPS / 4 * 32);
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    mbar_init(smem_u32(&ctl->never), 1);
    ctl->abort_flag = 0;
    ctl->no_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // both CTAs of a pair read the same group sizes, so they leave here together
  if (ctl->err) {
    if (threadIdx.x == 0) raise_error(&g_err, MOE_DEVERR_GROUP_SIZES);
    return;
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(smem_u32(&ctl->tmem_base), C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&ctl->tmem_base), C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  tc_fence_before();
  // a pair: the peer's barriers are initialised and its columns allocated
  // before any operand, commit or release crosses between the two CTAs
  if (PAIR) cluster_sync_all(); else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  if (PAIR && rank == 1 && threadIdx.x == 0 &&
      ld_shared_cluster_u32(mapa_shared(smem_u32(&ctl->tmem_base), 0)) != tmem_base)
    raise_error(&g_err, MOE_DEVERR_TMEM);  // the pair's accumulators would not line up
  const int total = ctl->total_tiles;
  volatile int* abort_flag = &ctl->abort_flag;
  bool timed_out = false;
  // release of accumulator `a` by one epilogue warp (to the pair's even CTA;
  // relaxed: it orders only tensor-memory loads that have already completed)
  auto release_acc = [&](uint32_t a) {
    if (PAIR)
      mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&ctl->tempty[a]), 0));
    else
      mbar_arrive(smem_u32(&ctl->tempty[a]));
  };

  // Roles: the control warps (producer, MMA issuer, and for promotion two
  // idle warps) and the epilogue warps.  With promotion each role's register
  // budget is set at the top of its own branch (a budget set before a join
  // would bind the code after it to the smaller one).
  if (warp < C::CTRL_WARPS) {
  if (C::SPLIT) setmaxnreg_dec<C::CTRL_REGS>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = 0;
      const bool w_blk = C::PROMOTE && p.rhs_mode == MOE_SCALE_PER_ROW_BLOCK128;
      for (int t = unit0; t < total && !timed_out; t += units) {
        const Tile tl = get_tile<MODE, PAIR>(p, ctl, t, rank);
        // promotion: bytes of this tile's weight-scale row per K block (a
        // narrower last N tile copies only its columns)
        const uint32_t sw_bytes = !w_blk ? 0u
                                  : (MODE == kPromoteSwiglu ? 2u * 128u * 4u
                                                            : static_cast<uint32_t>(min(BN, p.N - tl.n0)) * 4u);
        for (int kb = 0; kb < tl.nkb; ++kb) {
          const int s = it % NSTAGE;
          const uint32_t ph = (it / NSTAGE) & 1;
          const uint32_t q = it % kSwSlots;
          if (w_blk &&
              !CTRL_WAIT(smem_u32(&ctl->sempty[q]), ((it / kSwSlots) & 1) ^ 1, abort_flag, kWaitLimitNs)) {
            timed_out = true;
            break;
          }
          if (!CTRL_WAIT(smem_u32(&ctl->empty[s]), ph ^ 1, abort_flag, kWaitLimitNs)) {
            timed_out = true;
            break;
          }
          const uint32_t sa = base + s * STAGE_BYTES;
          if (PAIR) {
            // both CTAs' boxes complete on the even CTA's full barrier
            const uint32_t fb = mapa_shared(smem_u32(&ctl->full[s]), 0);
            if (rank == 0) mbar_arrive_expect_tx(smem_u32(&ctl->full[s]), C::TX_BYTES);
            tma_load_2d_pair(sa, &tmA, tl.ax + kb * C::KSTEP, tl.ay, fb);
            tma_load_2d_pair(sa + A_BYTES, &tmB, tl.bx + kb * C::KSTEP, tl.by, fb);
          } else {
            const uint32_t fb = smem_u32(&ctl->full[s]);
            mbar_arrive_expect_tx(fb, C::TX_BYTES);
            tma_load_2d(sa, &tmA, tl.ax + kb * C::KSTEP, tl.ay, fb);
            if (MODE == kSwiglu || MODE == kPromoteSwiglu || MODE == kMxSwiglu) {
              // B rows 0..127: wi_0 channels; rows 128..255: the matching wi_1 channels
              tma_load_2d(sa + A_BYTES, &tmB, tl.bx + kb * C::KSTEP, tl.by, fb);
              tma_load_2d(sa + 2 * A_BYTES, &tmB, tl.bx + kb * C::KSTEP, tl.by + p.F, fb);
            } else {
              tma_load_2d(sa + A_BYTES, &tmB, tl.bx + kb * C::KSTEP, tl.by, fb);
            }
            if (w_blk) {
              // the K block's weight-scale row, into ring slot q (the
              // epilogue waits for it on its own barrier)
              const uint32_t sb = smem_u32(&ctl->sfull[q]);
              mbar_arrive_expect_tx(sb, sw_bytes);
              const float* row = p.rhs_scale + (static_cast<int64_t>(tl.el) * p.kblocks + kb) * p.N;
              const uint32_t dst = smem_u32(sw_ring + q * BN);
              if (MODE == kPromoteSwiglu) {
                bulk_load(dst, row + tl.n0, 128 * 4, sb);                  // wi_0 channels of the tile
                bulk_load(dst + 128 * 4, row + p.F + tl.n0, 128 * 4, sb);  // the matching wi_1 channels
              } else {
                bulk_load(dst, row + tl.n0, sw_bytes, sb);
              }
            }
          }
          ++it;
        }
      }
      if (timed_out) {
        *abort_flag = 1;
        ctl->err = 2;
        // let the loads already issued land before the CTA can exit (the
        // full barriers that count them are this CTA's unless it is the
        // odd CTA of a pair)
        if (!PAIR || rank == 0)
          for (uint32_t j = (it > NSTAGE ? it - NSTAGE : 0); j < it; ++j)
            mbar_wait_bounded(smem_u32(&ctl->full[j % NSTAGE]), (j / NSTAGE) & 1, &ctl->no_abort, kWaitLimitNs);
        if (w_blk)  // and the scale rows
          for (uint32_t j = (it > kSwSlots ? it - kSwSlots : 0); j < it; ++j)
            mbar_wait_bounded(smem_u32(&ctl->sfull[j % kSwSlots]), (j / kSwSlots) & 1, &ctl->no_abort, kWaitLimitNs);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && (!PAIR || rank == 0)) {
      uint32_t it = 0, acc = 0;
      for (int t = unit0; t < total && !timed_out; t += units) {
        const Tile tl = get_tile<MODE, PAIR>(p, ctl, t, rank);
        if (tl.nkb == 0) continue;
        uint32_t a = acc % NACC;
        if (!C::PROMOTE) {
          if (!CTRL_WAIT(smem_u32(&ctl->tempty[a]), ((acc / NACC) & 1) ^ 1, abort_flag, kWaitLimitNs)) {
            timed_out = true;
            break;
          }
          tc_fence_after();
        }
        for (int kb = 0; kb < tl.nkb; ++kb) {
          if (C::PROMOTE) {
            a = acc % NACC;
            if (!CTRL_WAIT(smem_u32(&ctl->tempty[a]), ((acc / NACC) & 1) ^ 1, abort_flag, kWaitLimitNs)) {
              timed_out = true;
              break;
            }
            tc_fence_after();
          }
          const int s = it % NSTAGE;
          const uint32_t ph = (it / NSTAGE) & 1;
          const uint32_t q = it % kMxSfSlots;  // MXFP8: scale slot
          if (!CTRL_WAIT(smem_u32(&ctl->full[s]), ph, abort_flag, kWaitLimitNs) ||
              (C::MX && !CTRL_WAIT(smem_u32(&ctl->sffull[q]), (it / kMxSfSlots) & 1, abort_flag, kWaitLimitNs))) {
            timed_out = true;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + s * STAGE_BYTES;
          const uint64_t da = smem_desc_sw128(sa);
          const uint64_t db = smem_desc_sw128(sa + A_BYTES);
          // kSplit: K blocks [0, kb_split) accumulate into the tile's first
          // accumulator, the rest into its second (each segment starts fresh)
          const bool seg1 = MODE == kSplit && kb >= p.kb_split;
          const uint32_t d_tmem = tmem_base + a * BN * C::SEGS + (seg1 ? BN : 0);
          const int seg_kb0 = seg1 ? p.kb_split : 0;
          // MXFP8: the stage's scale atoms into its tensor-memory slot (A: 4
          // columns, B: 8), ahead of the MMAs that read them
          const uint32_t sfa_t = tmem_base + C::SF_COL0 + 16 * s, sfb_t = sfa_t + 4;
          if (C::MX) {
            const uint32_t sf_sm = sf_ring + q * kMxSfStageBytes;
            tmem_cp_32x128b_warpx4(sfa_t, smem_desc_plain(sf_sm));
            tmem_cp_32x128b_warpx4(sfb_t, smem_desc_plain(sf_sm + 512));
            tmem_cp_32x128b_warpx4(sfb_t + 4, smem_desc_plain(sf_sm + 1024));
          }
#pragma unroll
          for (int k4 = 0; k4 < BK / UMMA_K; ++k4) {
            const uint32_t accumulate = C::PROMOTE ? (k4 > 0) : (kb > seg_kb0 || k4 > 0);
            // +32 bytes along K inside the 128-byte swizzled row = +2 in the
            // descriptor's address field (16-byte units)
            if (C::MX)  // K block k4 of the stage: byte k4 of every scale cell
              mma_mx(d_tmem, da + 2 * k4, db + 2 * k4, idesc_mx_e4m3(BM, BN, k4, k4), sfa_t, sfb_t, accumulate);
            else if (C::BF)
              mma_bf16(d_tmem, da + 2 * k4, db + 2 * k4, IDESC, accumulate);
            else if (PAIR)
              mma_f8_pair(d_tmem, da + 2 * k4, db + 2 * k4, IDESC, accumulate);
            else
              mma_f8(d_tmem, da + 2 * k4, db + 2 * k4, IDESC, accumulate);
          }
          if (PAIR)
            mma_commit_pair_mc(smem_u32(&ctl->empty[s]), 0x3);  // frees the stage in both CTAs
          else
            mma_commit(smem_u32(&ctl->empty[s]));
          if (C::MX) mma_commit(smem_u32(&ctl->sfempty[q]));  // and the scale slot
          if (C::PROMOTE) {
            mma_commit(smem_u32(&ctl->tfull[a]));
            ++acc;
          }
          ++it;
        }
        if (timed_out) break;
        if (!C::PROMOTE) {
          if (PAIR)
            mma_commit_pair_mc(smem_u32(&ctl->tfull[a]), 0x3);
          else
            mma_commit(smem_u32(&ctl->tfull[a]));
          ++acc;
        }
      }
      // drain: every MMA this thread issued has completed once `drain` flips
      if (PAIR)
        mma_commit_pair(smem_u32(&ctl->drain));
      else
        mma_commit(smem_u32(&ctl->drain));
      if (!mbar_wait_bounded(smem_u32(&ctl->drain), 0, &ctl->no_abort, kWaitLimitNs)) timed_out = true;
      if (timed_out) {
        *abort_flag = 1;
        ctl->err = 2;
      }
    }
    __syncwarp();
  } else if (C::MX && warp == 2) {
    // ------------------------------------------------ MXFP8 scale gatherer
    // Each stage's E8M0 codes go into the stage's atoms by 4-byte cp.async
    // copies (lane l: tile rows 32 c + l): 4 A rows and 8 B rows a lane, the
    // word of a row holding the stage's four K blocks.  The codes are
    // K-block-major, so the words of a tile's rows for one stage are
    // adjacent and every copy instruction of the warp reads one 128-byte
    // line.  The atoms go to a ring of kMxSfSlots slots; a slot is free once
    // the MMAs that read its previous contents completed (sfempty, committed
    // by the MMA issuer).  A slot is announced (32 arrivals on sffull) LAG
    // stages later, once its copies have landed and been made visible to the
    // tensor core's (async-proxy) reads, so that each lane keeps LAG stages
    // of copies in flight; with more slots than LAG the announcements stay
    // ahead of the MMAs.
    constexpr uint32_t LAG = MOE_MX_LAG;
    static_assert(LAG >= 1 && LAG < kMxSfSlots, "the gatherer runs at most kMxSfSlots - 1 stages ahead");
    uint32_t it = 0;
    const uint32_t* lsf = reinterpret_cast<const uint32_t*>(p.lhs_sf);
    const uint32_t* rsf = reinterpret_cast<const uint32_t*>(p.rhs_sf);
    const int64_t brows = static_cast<int64_t>(p.El) * p.N;  // rows of the rhs (N = 2F for kMxSwiglu)
    for (int t = unit0; t < total && !timed_out; t += units) {
      const Tile tl = get_tile<MODE, PAIR>(p, ctl, t, rank);
      for (int kb = 0; kb < tl.nkb; ++kb) {
        const uint32_t q = it % kMxSfSlots;
        if (!CTRL_WAIT(smem_u32(&ctl->sfempty[q]), ((it / kMxSfSlots) & 1) ^ 1, abort_flag, kWaitLimitNs)) {
          timed_out = true;
          break;
        }
        const uint32_t dst = sf_ring + q * kMxSfStageBytes + lane * 16;
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // rows past M (end of the last group) read as zeros
          const int64_t row = static_cast<int64_t>(tl.row0) + 32 * c + lane;
          const bool ok = row < p.M;
          cp_async_4(dst + 4 * c, ok ? lsf + kb * p.M + row : lsf, ok ? 4u : 0u);
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int nl = 32 * c + lane;  // B row of the tile
          int64_t wrow;
          bool ok = true;
          if (MODE == kMxSwiglu) {  // rows 0..127: wi_0 channels; 128..255: the matching wi_1 channels
            wrow = static_cast<int64_t>(tl.el) * 2 * p.F + (nl < 128 ? tl.n0 + nl : p.F + tl.n0 + nl - 128);
          } else {  // channels past N (a narrower last N tile) read as zeros
            ok = tl.n0 + nl < p.N;
            wrow = static_cast<int64_t>(tl.el) * p.N + tl.n0 + nl;
          }
          cp_async_4(dst + 512 * (1 + (c >> 2)) + 4 * (c & 3), ok ? rsf + kb * brows + wrow : rsf, ok ? 4u : 0u);
        }
        cp_async_commit();
        if (it >= LAG) {
          cp_async_wait<LAG>();
          fence_proxy_async_smem();
          mbar_arrive(smem_u32(&ctl->sffull[(it - LAG) % kMxSfSlots]));
        }
        ++it;
      }
    }
    // the last LAG stages (and, after a timeout, every copy in flight)
    cp_async_wait<0>();
    fence_proxy_async_smem();
    for (uint32_t j = it > LAG ? it - LAG : 0; j < it; ++j) mbar_arrive(smem_u32(&ctl->sffull[j % kMxSfSlots]));
    if (timed_out) {
      *abort_flag = 1;
      ctl->err = 2;
    }
  }
  } else {
    if (C::SPLIT) setmaxnreg_inc<C::EPI_REGS>();
    // ------------------------------------------------------------ epilogue
    const int q4 = warp & 3;                            // TMEM lane quarter of this warp
    const int half = (warp - C::CTRL_WARPS) >> 2;  // column part of the warp (0 with 4 epilogue warps)
    const int r = q4 * 32 + lane;                       // row of the tile = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(q4 * 32) << 16;
    uint32_t acc = 0;
    uint32_t tcount = 0;  // promotion: tiles done by this CTA
    if (p.stall && !mbar_wait_bounded_warp(smem_u32(&ctl->never), 0, abort_flag, p.stall_ns)) timed_out = true;
    int stg_sel = 0;  // kTgmm: staging buffer of this warp's next block
    for (int t = unit0; t < total && !timed_out; t += units) {
      const Tile tl = get_tile<MODE, PAIR>(p, ctl, t, rank);
      const bool row_ok = r < tl.rows;
      if (MODE == kTgmm) {
        float* out = static_cast<float*>(p.out);
        const int64_t krow = tl.row0 + r;
        constexpr int WCOLS = BN / (EPI_WARPS / 4);  // columns of the tile this warp writes
        if (tl.nkb == 0) {
          // an expert with no rows: dW_e = 0; row by row, the warp's 32 lanes
          // cover its WCOLS columns (4 each) with one coalesced store per row
          static_assert(MODE != kTgmm || WCOLS == 128, "zero fill: 32 lanes x 4 columns");
          const int cz = tl.n0 + half * WCOLS + 4 * lane;
          float* zbase = out + (static_cast<int64_t>(tl.el) * p.K + tl.row0 + q4 * 32) * p.N + cz;
          const int zrows = min(32, tl.rows - q4 * 32);
          if (cz < p.N)
            for (int i = 0; i < zrows; ++i)
              *reinterpret_cast<float4*>(zbase + static_cast<int64_t>(i) * p.N) = make_float4(0.f, 0.f, 0.f, 0.f);
          continue;
        }
        const uint32_t a = acc % NACC;
        // the scales are requested first, so that their loads are in flight
        // while the accumulator is awaited; each block's column scales are
        // loaded while the block before it is written out
        const float sx = row_ok ? group_col_scale(p.lhs_scale, p.lhs_mode, tl.el, static_cast<int>(krow), p.K) : 0.f;
        const bool per_col = p.rhs_mode == MOE_SCALE_PER_GROUP_COL;
        const float* sgb = p.rhs_scale + (per_col ? static_cast<int64_t>(tl.el) * p.N : 0);
        const float sg_t = per_col ? 0.f : __ldg(p.rhs_scale);
        const bool block_rows = tl.rows - q4 * 32 > 0;  // rows >= K are clipped by the store
        constexpr int NB = WCOLS / 32;  // 32-column blocks of this warp
        const int cb0 = half * NB;
        float sgr[2][32];
        load_col_scales32(sgb, tl.n0 + cb0 * 32, p.N, per_col, sg_t, sgr[0]);
        if (!mbar_wait_bounded_warp(smem_u32(&ctl->tfull[a]), (acc / NACC) & 1, abort_flag, kWaitLimitNs)) {
          timed_out = true;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int i = 0; i < NB; ++i) {
          const int c = cb0 + i;
          const int nb = tl.n0 + c * 32;
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem_base + lane_addr + a * BN + c * 32, v);
          if (i + 1 < NB) load_col_scales32(sgb, nb + 32, p.N, per_col, sg_t, sgr[(i + 1) & 1]);
          const float* sg = sgr[i & 1];
          tmem_wait_ld();
          // this warp's 32x32 block, staged in the swizzled box layout and
          // written by one TMA store; the staging buffers rotate
          uint8_t* buf = stg_base + (warp - C::CTRL_WARPS) * C::STG_WARP_BYTES + stg_sel * 4096;
          if (lane == 0) bulk_wait_read<C::STG_BUFS - 1>();  // the store last issued from `buf` has read it
          __syncwarp();
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            float4 o;
            o.x = __uint_as_float(v[g * 4 + 0]) * sx * sg[g * 4 + 0];
            o.y = __uint_as_float(v[g * 4 + 1]) * sx * sg[g * 4 + 1];
            o.z = __uint_as_float(v[g * 4 + 2]) * sx * sg[g * 4 + 2];
            o.w = __uint_as_float(v[g * 4 + 3]) * sx * sg[g * 4 + 3];
            *reinterpret_cast<float4*>(buf + lane * 128 + ((g ^ (lane & 7)) << 4)) = o;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && block_rows && nb < p.N) {
            tma_store_3d(&tmO, smem_u32(buf), nb, tl.row0 + q4 * 32, tl.el);
            bulk_commit();
          }
          stg_sel = stg_sel + 1 == C::STG_BUFS ? 0 : stg_sel + 1;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release_acc(a);
        ++acc;
      } else if (MODE == kSwiglu) {
        // 8 warps: TMEM lane quarter q4, h columns [half*64, half*64 + 64) of
        // the tile; accumulator columns c*32.. hold a0, 128 + c*32.. hold a1.
        const int64_t row = static_cast<int64_t>(tl.row0) + r;
        const uint32_t a = acc % NACC;
        if (!mbar_wait_bounded_warp(smem_u32(&ctl->tfull[a]), (acc / NACC) & 1, abort_flag, kWaitLimitNs)) {
          timed_out = true;
          break;
        }
        tc_fence_after();
        const float sa = row_ok ? lhs_scale_at(p, row, 0) : 0.f;
        const bool per_chan = p.rhs_mode == MOE_SCALE_PER_ROW;
        const float* swb = p.rhs_scale + (per_chan ? static_cast<int64_t>(tl.el) * 2 * p.F : 0);
        float hs = 1.0f, hinv = 1.0f;
        if (p.h_mode == MOE_SCALE_PER_TENSOR) {
          hs = __ldg(p.h_static);
          hinv = __frcp_rn(hs);
        }
        float amax = 0.0f;
        uint32_t hp[32];  // this warp's 64 h values of the row, bf16 pairs (per-128 h scales)
        // four chunks of 16 h columns (16-column TMEM loads keep the live
        // arrays small enough to stay in registers)
        constexpr int CW = 16, NCH = 64 / CW;
#pragma unroll
        for (int cc = 0; cc < NCH; ++cc) {
          const int c = half * NCH + cc;  // chunk of the tile's 128 h columns
          uint32_t v0[CW], v1[CW];
          tmem_ld_32x32b_x16(tmem_base + lane_addr + a * BN + c * CW, v0);
          tmem_ld_32x32b_x16(tmem_base + lane_addr + a * BN + 128 + c * CW, v1);
          tmem_wait_ld();
          if (cc == NCH - 1) {  // the accumulator is no longer needed: release it early
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release_acc(a);
          }
          const int hc = tl.n0 + c * CW;  // first h column of the chunk
          float f0[CW], f1[CW], h[CW];
          uint32_t a0b[CW / 2], a1b[CW / 2], hb[CW / 2];  // the same values as packed bf16 pairs
          const uint64_t sa2 = f2_pack(sa, sa);
#pragma unroll
          for (int g = 0; g < CW / 4; ++g) {
            float4 s0, s1;
            if (per_chan) {
              s0 = __ldg(reinterpret_cast<const float4*>(swb + hc) + g);
              s1 = __ldg(reinterpret_cast<const float4*>(swb + p.F + hc) + g);
            } else {
              s0.x = s0.y = s0.z = s0.w = __ldg(swb);
              s1 = s0;
            }
            const float w0[4] = {s0.x, s0.y, s0.z, s0.w}, w1[4] = {s1.x, s1.y, s1.z, s1.w};
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              // a0, a1 rounded to bf16 exactly as gmm_fp8 stores them: bf16((acc * sa) * sw)
              const int j = g * 4 + 2 * jj;
              float x0, x1;
              f2_unpack(f2_mul(f2_mul(f2_pack(__uint_as_float(v0[j]), __uint_as_float(v0[j + 1])), sa2),
                               f2_pack(w0[2 * jj], w0[2 * jj + 1])),
                        x0, x1);
              a0b[j / 2] = pack_bf16x2(x0, x1);
              f0[j] = bf16lo(a0b[j / 2]);
              f0[j + 1] = bf16hi(a0b[j / 2]);
              f2_unpack(f2_mul(f2_mul(f2_pack(__uint_as_float(v1[j]), __uint_as_float(v1[j + 1])), sa2),
                               f2_pack(w1[2 * jj], w1[2 * jj + 1])),
                        x0, x1);
              a1b[j / 2] = pack_bf16x2(x0, x1);
              f1[j] = bf16lo(a1b[j / 2]);
              f1[j + 1] = bf16hi(a1b[j / 2]);
            }
          }
          swiglu_h_x2<CW>(f0, f1, h, hb);
#pragma unroll
          for (int j = 0; j < CW; ++j) amax = fmaxf(amax, fabsf(h[j]));
          if (row_ok) {
            if (p.a_out) {
              uint4* d0 = reinterpret_cast<uint4*>(p.a_out + row * 2 * p.F + hc);
              uint4* d1 = reinterpret_cast<uint4*>(p.a_out + row * 2 * p.F + p.F + hc);
#pragma unroll
              for (int g = 0; g < CW / 8; ++g) {
                d0[g] = make_uint4(a0b[4 * g], a0b[4 * g + 1], a0b[4 * g + 2], a0b[4 * g + 3]);
                d1[g] = make_uint4(a1b[4 * g], a1b[4 * g + 1], a1b[4 * g + 2], a1b[4 * g + 3]);
              }
            }
          }
          if (p.h_mode == MOE_SCALE_PER_TENSOR) {  // the chunk's codes (16 bytes) into hp[4 cc ..]
            float qv[CW];
            quant_n<CW>(h, hs, hinv, qv);
            const uint2 lo8 = pack_e4m3x8(qv), hi8 = pack_e4m3x8(qv + 8);
            hp[4 * cc] = lo8.x;
            hp[4 * cc + 1] = lo8.y;
            hp[4 * cc + 2] = hi8.x;
            hp[4 * cc + 3] = hi8.y;
          } else {
#pragma unroll
            for (int j = 0; j < CW / 2; ++j) hp[cc * (CW / 2) + j] = hb[j];
          }
        }
        // the warp's rows go out as whole row segments (warp_store_32x64B):
        // h bf16 [64 columns = 128 bytes] or codes [64 bytes] of each row
        uint8_t* stg = stg_base + (warp - C::CTRL_WARPS) * C::STG_WARP_BYTES;
        const int wrows = tl.rows - q4 * 32;
        const int64_t wrow0 = static_cast<int64_t>(tl.row0) + q4 * 32;
        const int hc0 = tl.n0 + half * 64;  // first h column of this warp
        if (p.h_mode == MOE_SCALE_PER_ROW) {
          uint8_t* hb0 = reinterpret_cast<uint8_t*>(p.h_out + wrow0 * p.F + hc0);
          warp_store_32x64B(stg, *reinterpret_cast<const uint32_t(*)[16]>(hp), hb0, 2 * static_cast<int64_t>(p.F),
                            wrows, 64);
          warp_store_32x64B(stg, *reinterpret_cast<const uint32_t(*)[16]>(hp + 16), hb0 + 64,
                            2 * static_cast<int64_t>(p.F), wrows, 64);
        } else if (p.h_mode == MOE_SCALE_PER_TENSOR) {
          warp_store_32x64B(stg, *reinterpret_cast<const uint32_t(*)[16]>(hp), p.h_q + wrow0 * p.F + hc0, p.F, wrows,
                            64);
        }
        const int par = acc & 1;
        ++acc;
        if (p.h_mode == MOE_SCALE_PER_ROW) {
          // non-negative floats order like their bit patterns
          if (row_ok) atomicMax(reinterpret_cast<unsigned int*>(p.h_scale) + row, __float_as_uint(amax));
        } else if (p.h_mode == MOE_SCALE_PER_ROW_BLOCK128) {
          // the tile's 128 h columns are one 128-column scale block, split
          // over the two warps of this lane quarter: exchange their maxima
          ctl->pamax[par][q4][half][lane] = amax;
          named_barrier_sync(1 + q4, 64);
          const float m = fmaxf(amax, ctl->pamax[par][q4][half ^ 1][lane]);
          const float sblk = absmax_scale(m);
          const float inv = __frcp_rn(sblk);
          if (row_ok && half == 0) p.h_scale[row * (p.F / 128) + tl.n0 / 128] = sblk;
          uint32_t cw[16];  // the 64 codes of this warp's part of the row
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            float x16[16], qv[16];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              x16[2 * j] = bf16lo(hp[g * 8 + j]);
              x16[2 * j + 1] = bf16hi(hp[g * 8 + j]);
            }
            quant_n<16>(x16, sblk, inv, qv);
            const uint2 lo8 = pack_e4m3x8(qv), hi8 = pack_e4m3x8(qv + 8);
            cw[4 * g] = lo8.x;
            cw[4 * g + 1] = lo8.y;
            cw[4 * g + 2] = hi8.x;
            cw[4 * g + 3] = hi8.y;
          }
          warp_store_32x64B(stg, cw, p.h_q + wrow0 * p.F + hc0, p.F, wrows, 64);
        }
      } else if (MODE == kSplit) {
        // out = bf16((s0 * acc0 + s1 * acc1) * s_a): the two K segments'
        // fp32 sums meet in the epilogue, each with its static weight scale
        uint16_t* out = static_cast<uint16_t*>(p.out);
        const int64_t row = static_cast<int64_t>(tl.row0) + r;
        const uint32_t a = acc % NACC;
        if (!mbar_wait_bounded_warp(smem_u32(&ctl->tfull[a]), (acc / NACC) & 1, abort_flag, kWaitLimitNs)) {
          timed_out = true;
          break;
        }
        tc_fence_after();
        const float sa = row_ok ? lhs_scale_at(p, row, 0) : 0.f;
        const float s0 = __ldg(p.rhs_scale), s1 = __ldg(p.rhs_scale + 1);
        const bool has0 = p.kb_split > 0, has1 = p.kb_split < p.kblocks;
        const uint32_t t0 = tmem_base + lane_addr + a * BN * C::SEGS;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          const int nb = tl.n0 + c * 32;
          uint32_t v0[32], v1[32];
          if (has0) tmem_ld_32x32b_x32(t0 + c * 32, v0);
          if (has1) tmem_ld_32x32b_x32(t0 + BN + c * 32, v1);
          tmem_wait_ld();
          float f[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float p0 = has0 ? __fmul_rn(__uint_as_float(v0[j]), s0) : 0.0f;
            f[j] = __fmul_rn(has1 ? __fmaf_rn(__uint_as_float(v1[j]), s1, p0) : p0, sa);
          }
          // stage this warp's 32x32 bf16 block, then write 8 rows (64 contiguous bytes each) per instruction
          uint8_t* stg = stg_base + (warp - C::CTRL_WARPS) * C::STG_WARP_BYTES;
#pragma unroll
          for (int g = 0; g < 4; ++g)
            *reinterpret_cast<uint4*>(stg + lane * C::STG_PITCH + 16 * g) =
                make_uint4(pack_bf16x2(f[8 * g], f[8 * g + 1]), pack_bf16x2(f[8 * g + 2], f[8 * g + 3]),
                           pack_bf16x2(f[8 * g + 4], f[8 * g + 5]), pack_bf16x2(f[8 * g + 6], f[8 * g + 7]));
          __syncwarp();
          const int seg = (lane & 3) * 8;  // bf16 column offset of this lane's 16 bytes
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int rr = i * 8 + (lane >> 2);
            const int64_t orow = static_cast<int64_t>(tl.row0) + q4 * 32 + rr;
            if (rr < tl.rows - q4 * 32 && nb + seg < p.N)
              *reinterpret_cast<uint4*>(out + orow * p.N + nb + seg) =
                  *reinterpret_cast<const uint4*>(stg + rr * C::STG_PITCH + 2 * seg);
          }
          __syncwarp();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release_acc(a);
        ++acc;
      } else if (MODE == kFinal) {
        uint16_t* out = static_cast<uint16_t*>(p.out);
        const int64_t row = static_cast<int64_t>(tl.row0) + r;
        const uint32_t a = acc % NACC;
        if (!mbar_wait_bounded_warp(smem_u32(&ctl->tfull[a]), (acc / NACC) & 1, abort_flag, kWaitLimitNs)) {
          timed_out = true;
          break;
        }
        tc_fence_after();
        const float sa = row_ok ? lhs_scale_at(p, row, 0) : 0.f;
        // channel scales: branch on the mode once per tile, then 16-byte
        // broadcast loads (every lane reads the same 32 scales)
        const bool per_chan = p.rhs_mode == MOE_SCALE_PER_ROW;
        const float* swb = p.rhs_scale + (per_chan ? static_cast<int64_t>(tl.el) * p.N : 0);
        const float sw_t = per_chan ? 0.f : __ldg(p.rhs_scale);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          const int nb = tl.n0 + c * 32;
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem_base + lane_addr + a * BN + c * 32, v);
          float sw[32];
          load_col_scales32(swb, nb, p.N, per_chan, sw_t, sw);
          tmem_wait_ld();
          // stage this warp's 32x32 bf16 block, then write 8 rows (64 contiguous bytes each) per instruction
          uint8_t* stg = stg_base + (warp - C::CTRL_WARPS) * C::STG_WARP_BYTES;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint4 q;
            q.x = pack_bf16x2(__fmul_rn(__fmul_rn(__uint_as_float(v[8 * g + 0]), sa), sw[8 * g + 0]),
                              __fmul_rn(__fmul_rn(__uint_as_float(v[8 * g + 1]), sa), sw[8 * g + 1]));
            q.y = pack_bf16x2(__fmul_rn(__fmul_rn(__uint_as_float(v[8 * g + 2]), sa), sw[8 * g + 2]),
                              __fmul_rn(__fmul_rn(__uint_as_float(v[8 * g + 3]), sa), sw[8 * g + 3]));
            q.z = pack_bf16x2(__fmul_rn(__fmul_rn(__uint_as_float(v[8 * g + 4]), sa), sw[8 * g + 4]),
                              __fmul_rn(__fmul_rn(__uint_as_float(v[8 * g + 5]), sa), sw[8 * g + 5]));
            q.w = pack_bf16x2(__fmul_rn(__fmul_rn(__uint_as_float(v[8 * g + 6]), sa), sw[8 * g + 6]),
                              __fmul_rn(__fmul_rn(__uint_as_float(v[8 * g + 7]), sa), sw[8 * g + 7]));
            *reinterpret_cast<uint4*>(stg + lane * C::STG_PITCH + 16 * g) = q;
          }
          __syncwarp();
          const int seg = (lane & 3) * 8;  // bf16 column offset of this lane's 16 bytes
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int rr = i * 8 + (lane >> 2);
            const int64_t orow = static_cast<int64_t>(tl.row0) + q4 * 32 + rr;
            if (rr < tl.rows - q4 * 32 && nb + seg < p.N)
              *reinterpret_cast<uint4*>(out + orow * p.N + nb + seg) =
                  *reinterpret_cast<const uint4*>(stg + rr * C::STG_PITCH + 2 * seg);
          }
          __syncwarp();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release_acc(a);
        ++acc;
      } else if (MODE == kMx) {
        // MXFP8: the scales were applied by the MMAs, so out = bf16(acc).
        // With one accumulator, the tile (8 warps: lane quarter q4, columns
        // [128 half, 128 half + 128)) is read into registers and released
        // before any store, so the next tile's MMAs run under the stores.
        // (Timing variants that skipped this wait, or these loads, ran no
        // faster: the single accumulator is not what bounds the kernel.)
        uint16_t* out = static_cast<uint16_t*>(p.out);
        if (!mbar_wait_bounded_warp(smem_u32(&ctl->tfull[0]), acc & 1, abort_flag, kWaitLimitNs)) {
          timed_out = true;
          break;
        }
        tc_fence_after();
        uint32_t v[4][32];
#pragma unroll
        for (int i = 0; i < 4; ++i) tmem_ld_32x32b_x32(tmem_base + lane_addr + half * 128 + 32 * i, v[i]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release_acc(0);
        ++acc;
        // the warp's 32 rows, one 32-column block at a time, as whole row
        // segments (rows past the group's end are not stored)
        uint8_t* stg = stg_base + (warp - C::CTRL_WARPS) * C::STG_WARP_BYTES;
        uint8_t* obase = reinterpret_cast<uint8_t*>(out + (static_cast<int64_t>(tl.row0) + q4 * 32) * p.N);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int nb = tl.n0 + half * 128 + 32 * i;
          if (nb < p.N) {  // the same for the whole warp
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(__uint_as_float(v[i][2 * j]), __uint_as_float(v[i][2 * j + 1]));
            warp_store_32x64B(stg, w, obase + 2 * nb, 2 * static_cast<int64_t>(p.N), tl.rows - q4 * 32,
                              2 * (p.N - nb));
          }
        }
      } else if (MODE == kMxSwiglu) {
        // MXFP8 wi gmm + SwiGLU + MXFP8 requantisation.  The accumulator
        // holds a0 (columns 0..127) and a1 (128..255) of 128 h columns; warp
        // part `half` takes h columns [64 half, 64 half + 64) of the tile,
        // i.e. two 32-column MX blocks, both inside this thread's row, so a
        // block's amax needs no exchange.  a0, a1 are rounded to bf16 as
        // gmm_fp8_mx stores them, h = bf16(silu(a0) a1), then per block
        // X = floor(log2 amax) - 8 and codes e4m3(h / 2^X).
        const int64_t row = static_cast<int64_t>(tl.row0) + r;
        if (!mbar_wait_bounded_warp(smem_u32(&ctl->tfull[0]), acc & 1, abort_flag, kWaitLimitNs)) {
          timed_out = true;
          break;
        }
        tc_fence_after();
        uint32_t v0[2][32], v1[2][32];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          tmem_ld_32x32b_x32(tmem_base + lane_addr + half * 64 + 32 * i, v0[i]);
          tmem_ld_32x32b_x32(tmem_base + lane_addr + 128 + half * 64 + 32 * i, v1[i]);
        }
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release_acc(0);
        ++acc;
        // this thread's 64 h codes (two MX blocks) go out with the warp's
        // other rows as whole row segments
        uint32_t codes[16];
        {
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int hc = tl.n0 + half * 64 + 32 * i;  // first h column of the block
            float f0[32], f1[32], h[32];
            uint32_t a0b[16], a1b[16], hb[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              a0b[j / 2] = pack_bf16x2(__uint_as_float(v0[i][j]), __uint_as_float(v0[i][j + 1]));
              a1b[j / 2] = pack_bf16x2(__uint_as_float(v1[i][j]), __uint_as_float(v1[i][j + 1]));
              f0[j] = bf16lo(a0b[j / 2]);
              f0[j + 1] = bf16hi(a0b[j / 2]);
              f1[j] = bf16lo(a1b[j / 2]);
              f1[j + 1] = bf16hi(a1b[j / 2]);
            }
            swiglu_h_x2<32>(f0, f1, h, hb);
            float amax = 0.0f;
#pragma unroll
            for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(h[j]));
            const int X = mx_shared_exp(amax);
            const float inv = mx_inv_scale(X);
#pragma unroll
            for (int j = 0; j < 32; ++j) h[j] = __fmul_rn(h[j], inv);  // exact: a power of two
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              const uint2 c8 = pack_e4m3x8(h + 8 * g);
              codes[8 * i + 2 * g] = c8.x;
              codes[8 * i + 2 * g + 1] = c8.y;
            }
            if (row_ok) p.h_sf[((hc >> 7) * p.M + row) * 4 + ((hc >> 5) & 3)] = static_cast<uint8_t>(X + 127);
            if (p.a_out && row_ok) {
              uint4* d0 = reinterpret_cast<uint4*>(p.a_out + row * 2 * p.F + hc);
              uint4* d1 = reinterpret_cast<uint4*>(p.a_out + row * 2 * p.F + p.F + hc);
#pragma unroll
              for (int g = 0; g < 4; ++g) {
                d0[g] = make_uint4(a0b[4 * g], a0b[4 * g + 1], a0b[4 * g + 2], a0b[4 * g + 3]);
                d1[g] = make_uint4(a1b[4 * g], a1b[4 * g + 1], a1b[4 * g + 2], a1b[4 * g + 3]);
              }
            }
          }
        }
        uint8_t* stg = stg_base + (warp - C::CTRL_WARPS) * C::STG_WARP_BYTES;
        warp_store_32x64B(stg, codes, p.h_q + (static_cast<int64_t>(tl.row0) + q4 * 32) * p.F + tl.n0 + half * 64,
                          p.F, tl.rows - q4 * 32, 64);
      } else if (MODE == kBf16) {
        // plain bf16 contraction without scales: bf16 rows staged through
        // shared memory as in the fp8 gmm, or fp32 rows written directly
        const int64_t row = static_cast<int64_t>(tl.row0) + r;
        const uint32_t a = acc % NACC;
        if (!mbar_wait_bounded_warp(smem_u32(&ctl->tfull[a]), (acc / NACC) & 1, abort_flag, kWaitLimitNs)) {
          timed_out = true;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          const int nb = tl.n0 + c * 32;
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem_base + lane_addr + a * BN + c * 32, v);
          tmem_wait_ld();
          if (p.out_f32) {
            float* out = static_cast<float*>(p.out);
#pragma unroll
            for (int h = 0; h < 2; ++h)  // N is a multiple of 16: each 16 columns are all in range or all past N
              if (row_ok && nb + 16 * h < p.N)
#pragma unroll
                for (int g = 0; g < 4; ++g)
                  *reinterpret_cast<float4*>(out + row * p.N + nb + 16 * h + 4 * g) =
                      make_float4(__uint_as_float(v[16 * h + 4 * g]), __uint_as_float(v[16 * h + 4 * g + 1]),
                                  __uint_as_float(v[16 * h + 4 * g + 2]), __uint_as_float(v[16 * h + 4 * g + 3]));
          } else {
            uint16_t* out = static_cast<uint16_t*>(p.out);
            uint8_t* stg = stg_base + (warp - C::CTRL_WARPS) * C::STG_WARP_BYTES;
#pragma unroll
            for (int g = 0; g < 4; ++g)
              *reinterpret_cast<uint4*>(stg + lane * C::STG_PITCH + 16 * g) =
                  make_uint4(pack_bf16x2(__uint_as_float(v[8 * g]), __uint_as_float(v[8 * g + 1])),
                             pack_bf16x2(__uint_as_float(v[8 * g + 2]), __uint_as_float(v[8 * g + 3])),
                             pack_bf16x2(__uint_as_float(v[8 * g + 4]), __uint_as_float(v[8 * g + 5])),
                             pack_bf16x2(__uint_as_float(v[8 * g + 6]), __uint_as_float(v[8 * g + 7])));
            __syncwarp();
            const int seg = (lane & 3) * 8;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int rr = i * 8 + (lane >> 2);
              const int64_t orow = static_cast<int64_t>(tl.row0) + q4 * 32 + rr;
              if (rr < tl.rows - q4 * 32 && nb + seg < p.N)
                *reinterpret_cast<uint4*>(out + orow * p.N + nb + seg) =
                    *reinterpret_cast<const uint4*>(stg + rr * C::STG_PITCH + 2 * seg);
            }
            __syncwarp();
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release_acc(a);
        ++acc;
      } else if (MODE == kRouter) {
        // the gate's logits of one token per thread (TMEM lane = row): the
        // logits to memory, then the softmax over the first E columns in
        // fp32 -- m = max, e_i = exp(l_i - m), Z summed in ascending i,
        // p_i = e_i / Z -- and the top-k by probability with ties to the
        // lower expert index, kept as a sorted list in registers
        const int64_t row = static_cast<int64_t>(tl.row0) + r;
        const uint32_t a = acc % NACC;
        if (!mbar_wait_bounded_warp(smem_u32(&ctl->tfull[a]), (acc / NACC) & 1, abort_flag, kWaitLimitNs)) {
          timed_out = true;
          break;
        }
        tc_fence_after();
        const int E = p.rE;
        const int nch = (E + 31) / 32;
        const uint32_t tb = tmem_base + lane_addr + a * BN;
        float mx = -INFINITY;
#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tb + 32 * c, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = 32 * c + j;
            const float l = __uint_as_float(v[j]);
            if (col < E) {
              mx = fmaxf(mx, l);
              if (row_ok) p.logits[row * E + col] = l;
            }
          }
        }
        float z = 0.0f;
#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tb + 32 * c, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (32 * c + j < E) z = __fadd_rn(z, exp_f32(__fsub_rn(__uint_as_float(v[j]), mx)));
        }
        constexpr int KMAX = 8;
        float tp[KMAX];
        int ti[KMAX];
#pragma unroll
        for (int s = 0; s < KMAX; ++s) {
          tp[s] = -1.0f;  // below every probability
          ti[s] = 0x7fffffff;
        }
#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tb + 32 * c, v);
          tmem_wait_ld();
          if (c == nch - 1) {  // the accumulator is in registers for the last time
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release_acc(a);
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = 32 * c + j;
            if (col >= E) continue;
            float cp = __fdiv_rn(exp_f32(__fsub_rn(__uint_as_float(v[j]), mx)), z);
            int ci = col;
            // insertion into the sorted list: larger probability first, the
            // lower index first among equal ones (a displaced entry carries
            // its own index down)
#pragma unroll
            for (int s = 0; s < KMAX; ++s) {
              const bool better = cp > tp[s] || (cp == tp[s] && ci < ti[s]);
              const float tf = better ? tp[s] : cp;
              const int tq = better ? ti[s] : ci;
              tp[s] = better ? cp : tp[s];
              ti[s] = better ? ci : ti[s];
              cp = tf;
              ci = tq;
            }
          }
        }
        if (row_ok)
#pragma unroll
          for (int s = 0; s < KMAX; ++s)
            if (s < p.rk) {
              p.topk_ids[row * p.rk + s] = ti[s];
              p.topk_w[row * p.rk + s] = tp[s];
            }
        ++acc;
      } else {
        // promotion (a blockwise operand scale): K block kb of the tile lands
        // in accumulator kb % 2 (the MMA runs one block ahead of this fold).
        // The epilogue warps fold it into fp32 registers: TMEM lane quarter
        // q4 (32 rows) x WC of the tile's 256 columns per warp -- plain gmm,
        // columns [WC part, +WC); fused SwiGLU, the a0 columns [WC/2 part,
        // +WC/2) and the matching a1 columns 128 + [WC/2 part, +WC/2).  Per
        // element and K block: acc += (p * s_w[n]) * s_a[m] on packed fp32
        // pairs, with s_w from the scale row the producer copied in with the
        // block's operands; a scale constant along K is applied at the end.
        constexpr bool SWG = MODE == kPromoteSwiglu;
        constexpr int NPART = EPI_WARPS / 4;  // warps per lane quarter
        constexpr int WC = BN / NPART;        // accumulator columns per warp
        constexpr int CWID = MOE_PROMOTE_CHUNK;  // columns per TMEM load
        constexpr int NCH = WC / CWID;           // chunks per warp
        constexpr bool DBUF = NPART == 1 || NPART == 2;  // double-buffered chunk loads (room in registers)
        const int part = half;
        const int64_t row = static_cast<int64_t>(tl.row0) + r;
        const bool a_blk = p.lhs_mode == MOE_SCALE_PER_ROW_BLOCK128;
        const bool w_blk = p.rhs_mode == MOE_SCALE_PER_ROW_BLOCK128;
        const int64_t srow = row_ok ? row : 0;
        const float* sab = p.lhs_scale + (a_blk ? srow * p.kblocks : 0);
        auto ccol = [&](int c) -> int {  // first accumulator column of this warp's chunk c
          return SWG ? (c < NCH / 2 ? (WC / 2) * part + CWID * c : 128 + (WC / 2) * part + CWID * (c - NCH / 2))
                     : WC * part + CWID * c;
        };
        // first accumulator column of 16-column group g of this warp (for the tails)
        auto gcol = [&](int g) -> int {
          return SWG ? (g < WC / 32 ? (WC / 2) * part + 16 * g : 128 + (WC / 2) * part + 16 * (g - WC / 32))
                     : WC * part + 16 * g;
        };
        uint64_t acc2[WC / 2];
#pragma unroll
        for (int j = 0; j < WC / 2; ++j) acc2[j] = 0ull;
        // the row's activation scale of the next K block is requested while
        // this block is folded (a block's fold outlasts the load's latency)
        auto load_a = [&](int kb) -> float { return (a_blk && kb < tl.nkb) ? __ldg(sab + kb) : 1.0f; };
        float sa_next = load_a(0);
        // the block loop, specialised by the operand(s) with a blockwise scale
        auto run = [&](auto fm_tag) {
          constexpr int FM = decltype(fm_tag)::value;  // 1: activations, 2: weights, 3: both
          auto fold16 = [&](const uint64_t* v, int c, const float* sw, uint64_t sa2) {  // one chunk of column pairs
#pragma unroll
            for (int j = 0; j < CWID / 4; ++j) {
              const uint64_t p0 = v[2 * j], p1 = v[2 * j + 1];
              uint64_t& c0 = acc2[(CWID / 2) * c + 2 * j];
              uint64_t& c1 = acc2[(CWID / 2) * c + 2 * j + 1];
              if (FM == 1) {
                c0 = f2_fma(p0, sa2, c0);
                c1 = f2_fma(p1, sa2, c1);
              } else {
                const float4 w4 = *reinterpret_cast<const float4*>(sw + ccol(c) + 4 * j);  // broadcast
                if (FM == 3) {
                  c0 = f2_fma(f2_mul(p0, f2_pack(w4.x, w4.y)), sa2, c0);
                  c1 = f2_fma(f2_mul(p1, f2_pack(w4.z, w4.w)), sa2, c1);
                } else {
                  c0 = f2_fma(p0, f2_pack(w4.x, w4.y), c0);
                  c1 = f2_fma(p1, f2_pack(w4.z, w4.w), c1);
                }
              }
            }
          };
          auto release = [&](uint32_t a) {  // every chunk of accumulator a is in registers
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[a]));
          };
#pragma unroll 1
          for (int kb = 0; kb < tl.nkb; ++kb) {
            const float sa = sa_next;
            sa_next = load_a(kb + 1);
            const uint32_t a = acc % NACC;
            const uint32_t q = acc % kSwSlots;
            // per-lane waits here, once per K block (a warp vote on each cost
            // 2 % of this kernel): the converged warp's lanes read the same
            // barrier phase, abort flag and timer in each instruction of the
            // wait loop, so they leave it together
            if (!mbar_wait_bounded(smem_u32(&ctl->tfull[a]), (acc / NACC) & 1, abort_flag, kWaitLimitNs) ||
                (FM != 1 &&
                 !mbar_wait_bounded(smem_u32(&ctl->sfull[q]), (acc / kSwSlots) & 1, abort_flag, kWaitLimitNs))) {
              timed_out = true;
              break;
            }
            tc_fence_after();
            const float* sw = sw_ring + q * BN;
            const uint64_t sa2 = f2_pack(sa, sa);
            const uint32_t tb = tmem_base + lane_addr + a * BN;
            static_assert(CWID == 16 || CWID == 32, "promotion chunk width");
            auto ld = [&](int c, uint64_t* u) {
              tmem_ld_32x32b_x16_pairs(tb + ccol(c), *reinterpret_cast<uint64_t(*)[8]>(u));
              if (CWID == 32) tmem_ld_32x32b_x16_pairs(tb + ccol(c) + 16, *reinterpret_cast<uint64_t(*)[8]>(u + 8));
            };
            if (DBUF) {
              uint64_t u[2][CWID / 2];
              ld(0, u[0]);
              tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < NCH; ++c) {
                // the next chunk's load is in flight while this one is folded
                if (c + 1 < NCH) ld(c + 1, u[(c + 1) & 1]);
                fold16(u[c & 1], c, sw, sa2);
                tmem_wait_ld();
                if (c == NCH - 2) release(a);
              }
            } else {
#pragma unroll
              for (int c = 0; c < NCH; ++c) {
                uint64_t u[CWID / 2];
                ld(c, u);
                tmem_wait_ld();
                if (c == NCH - 1) release(a);
                fold16(u, c, sw, sa2);
              }
            }
            if (FM != 1) {  // this warp is done with the scale row
              // the row is refilled by a bulk copy (the async proxy): order
              // this warp's generic reads of it before that write
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_u32(&ctl->sempty[q]));
            }
            ++acc;
          }
        };
        if (a_blk && w_blk)
          run(std::integral_constant<int, 3>{});
        else if (w_blk)
          run(std::integral_constant<int, 2>{});
        else
          run(std::integral_constant<int, 1>{});
        if (timed_out) break;
        // scales constant along K: per row / per tensor for the activations,
        // per channel / per tensor for the weights (1 for a blockwise side)
        const float sa_end = a_blk ? 1.0f
                                   : (row_ok ? (p.lhs_mode == MOE_SCALE_PER_ROW ? __ldg(p.lhs_scale + row)
                                                                                 : __ldg(p.lhs_scale))
                                             : 0.0f);
        const bool w_col = p.rhs_mode == MOE_SCALE_PER_ROW;
        const float* swb = p.rhs_scale + (w_col ? static_cast<int64_t>(tl.el) * p.N : 0);
        const float sw_t = (w_blk || w_col) ? 1.0f : __ldg(p.rhs_scale);
        // 8 output values (half h8 of 16-column group g) as gmm_fp8 stores
        // them: bf16((acc s_a) s_w)
        auto vals8 = [&](int g, int h8, float* f) {
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int q = 2 * h8 + i;  // 4-column quad of the group
            float4 w4 = make_float4(sw_t, sw_t, sw_t, sw_t);
            if (w_col) {
              // SwiGLU tiles: accumulator columns 0..127 are wi_0 channels
              // n0 + [0, 128), columns 128..255 wi_1 channels F + n0 + [0, 128)
              const int cc = gcol(g);
              const int ch = SWG ? (cc < 128 ? tl.n0 + cc : p.F + tl.n0 + cc - 128) : tl.n0 + cc;
              w4 = __ldg(reinterpret_cast<const float4*>(swb + ch) + q);
            }
            float x0, x1, x2, x3;
            f2_unpack(acc2[8 * g + 2 * q], x0, x1);
            f2_unpack(acc2[8 * g + 2 * q + 1], x2, x3);
            f[4 * i] = __fmul_rn(__fmul_rn(x0, sa_end), w4.x);
            f[4 * i + 1] = __fmul_rn(__fmul_rn(x1, sa_end), w4.y);
            f[4 * i + 2] = __fmul_rn(__fmul_rn(x2, sa_end), w4.z);
            f[4 * i + 3] = __fmul_rn(__fmul_rn(x3, sa_end), w4.w);
          }
        };
        if (!SWG) {
          // direct 16-byte stores of each thread's row: the tail runs on the
          // epilogue warps, the bound of this kernel, and staging the rows
          // for whole-sector stores was measured slower here (5.43 against
          // 5.03 ms on the DeepSeek-V3 wi contraction)
          if (row_ok) {
            uint16_t* out = static_cast<uint16_t*>(p.out);
#pragma unroll
            for (int c = 0; c < WC / 16; ++c) {
              const int nb = tl.n0 + gcol(c);  // N is a multiple of 16: the group is all in range or all past N
              if (nb < p.N) {
                uint32_t pk[8];
#pragma unroll
                for (int g = 0; g < 4; ++g) {  // 4 columns at a time, straight to bf16 pairs
                  float4 w4 = make_float4(sw_t, sw_t, sw_t, sw_t);
                  if (w_col) w4 = __ldg(reinterpret_cast<const float4*>(swb + nb) + g);
                  float x0, x1, x2, x3;
                  f2_unpack(acc2[8 * c + 2 * g], x0, x1);
                  f2_unpack(acc2[8 * c + 2 * g + 1], x2, x3);
                  pk[2 * g] = pack_bf16x2(__fmul_rn(__fmul_rn(x0, sa_end), w4.x), __fmul_rn(__fmul_rn(x1, sa_end), w4.y));
                  pk[2 * g + 1] =
                      pack_bf16x2(__fmul_rn(__fmul_rn(x2, sa_end), w4.z), __fmul_rn(__fmul_rn(x3, sa_end), w4.w));
                }
                uint16_t* dst = out + row * p.N + nb;
                *reinterpret_cast<uint4*>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *reinterpret_cast<uint4*>(dst + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
              }
            }
          }
        } else {
          // fused SwiGLU: this thread holds a0 and a1 of the h columns
          // n0 + (WC/2) part + [0, WC/2) of its row; h = bf16(silu(a0) a1) and
          // its codes as moe_swiglu_quant makes them from the stored a
          constexpr int HC = WC / 2;  // h columns of this warp
          float hs = 1.0f, hinv = 1.0f;
          if (p.h_mode == MOE_SCALE_PER_TENSOR) {
            hs = __ldg(p.h_static);
            hinv = __frcp_rn(hs);
          }
          float amax = 0.0f;
          uint32_t hp[HC / 2];  // the h values as bf16 pairs (per-128 h scales)
#pragma unroll
          for (int s8 = 0; s8 < HC / 8; ++s8) {  // 8 h columns at a time (few live temporaries)
            const int g = s8 >> 1, h8 = s8 & 1;  // 16-column group of a0 (a1: group g + WC / 32)
            float f0[8], f1[8], h[8];
            uint32_t hb[4], a0b[4], a1b[4];
            vals8(g, h8, f0);
            vals8(g + WC / 32, h8, f1);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              a0b[j] = pack_bf16x2(f0[2 * j], f0[2 * j + 1]);
              a1b[j] = pack_bf16x2(f1[2 * j], f1[2 * j + 1]);
              f0[2 * j] = bf16lo(a0b[j]);
              f0[2 * j + 1] = bf16hi(a0b[j]);
              f1[2 * j] = bf16lo(a1b[j]);
              f1[2 * j + 1] = bf16hi(a1b[j]);
            }
            swiglu_h_x2<8>(f0, f1, h, hb);
#pragma unroll
            for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(h[j]));
            const int hc = tl.n0 + HC * part + 8 * s8;  // first h column of the step
            if (row_ok) {
              if (p.a_out) {
                *reinterpret_cast<uint4*>(p.a_out + row * 2 * p.F + hc) = make_uint4(a0b[0], a0b[1], a0b[2], a0b[3]);
                *reinterpret_cast<uint4*>(p.a_out + row * 2 * p.F + p.F + hc) =
                    make_uint4(a1b[0], a1b[1], a1b[2], a1b[3]);
              }
              if (p.h_mode == MOE_SCALE_PER_ROW) {
                *reinterpret_cast<uint4*>(p.h_out + row * p.F + hc) = make_uint4(hb[0], hb[1], hb[2], hb[3]);
              } else if (p.h_mode == MOE_SCALE_PER_TENSOR) {
                float qv[8];
                quant_n<8>(h, hs, hinv, qv);
                *reinterpret_cast<uint2*>(p.h_q + row * p.F + hc) = pack_e4m3x8(qv);
              }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) hp[s8 * 4 + j] = hb[j];
          }
          const int par = tcount & 1;
          if (p.h_mode == MOE_SCALE_PER_ROW) {
            // non-negative floats order like their bit patterns
            if (row_ok) atomicMax(reinterpret_cast<unsigned int*>(p.h_scale) + row, __float_as_uint(amax));
          } else if (p.h_mode == MOE_SCALE_PER_ROW_BLOCK128) {
            // the tile's 128 h columns are one 128-column scale block, split
            // over the NPART warps of this lane quarter: they exchange their
            // maxima (a bounded wait on a barrier of those warps; the two
            // parities alternate between tiles)
            ctl->pamax[par][q4][part][lane] = amax;
            mbar_arrive(smem_u32(&ctl->xbar[q4][par]));
            if (!mbar_wait_bounded_warp(smem_u32(&ctl->xbar[q4][par]), (tcount >> 1) & 1, abort_flag, kWaitLimitNs)) {
              timed_out = true;
              break;
            }
            float m = amax;
#pragma unroll
            for (int o = 0; o < NPART; ++o) m = fmaxf(m, ctl->pamax[par][q4][o][lane]);
            if (row_ok) {
              const float sblk = absmax_scale(m);
              const float inv = __frcp_rn(sblk);
              if (part == 0) p.h_scale[row * (p.F / 128) + tl.n0 / 128] = sblk;
              float x16[16], qv[16];
              uint4* dst = reinterpret_cast<uint4*>(p.h_q + row * p.F + tl.n0 + HC * part);
#pragma unroll
              for (int g = 0; g < HC / 16; ++g) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  x16[2 * j] = bf16lo(hp[g * 8 + j]);
                  x16[2 * j + 1] = bf16hi(hp[g * 8 + j]);
                }
                quant_n<16>(x16, sblk, inv, qv);
                const uint2 lo8 = pack_e4m3x8(qv), hi8 = pack_e4m3x8(qv + 8);
                dst[g] = make_uint4(lo8.x, lo8.y, hi8.x, hi8.y);
              }
            }
          }
        }
        ++tcount;
      }
    }
    if (timed_out) {
      *abort_flag = 1;
      ctl->err = 2;
    }
    if (MODE == kTgmm && lane == 0) bulk_wait_all();  // the output stores have landed
  }

  tc_fence_before();
  // a pair: neither CTA leaves (or frees its columns) while the other may
  // still write its tensor memory or arrive on its barriers
  if (PAIR) cluster_sync_all(); else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
  if (threadIdx.x == 0 && ctl->err) raise_error(&g_err, MOE_DEVERR_TIMEOUT);
}

// ---- int8 weights (gmm_fp8_w8) ---------------------------------------------
// out[m, n] = s_x s_w sum_k e4m3(x)[m, k] q[g(m), n, k] in bf16: gmm_fp8 with
// the other weight type of "Keep qwix out of tpu-inference's fused MoE
// kernel and pre-quantize weights" (int8 codes with [E, blocks, 1, N]
// scales).  No tcgen05 MMA kind multiplies e4m3 by int8, but f16 holds every
// e4m3 value and every integer in [-127, 127] exactly, so both operands are
// converted to f16 on the SM and contracted by tcgen05.mma kind::f16 with
// fp32 accumulation:
//   - the weights are the A operand, read from tensor memory: four warps per
//     128 channels turn each stage's int8 rows into f16 (the byte under the
//     exponent of 1024 + 128, then one f16 subtraction) and store them with
//     tcgen05.st, so the converted weights never pass through shared memory;
//   - the activations are the B operand: one warp per 32 token rows turns
//     the stage's e4m3 rows into f16 (cvt.f16x2.e4m3x2) in the
//     128-byte-swizzled K-major layout the MMA reads from shared memory; or,
//     with XF16, a workspace already holds them as f16 (one HBM pass before
//     the kernel) and TMA lands them in that layout, so that per stage the
//     converters' reads and the f16 tile's writes leave shared memory.
// Two tile shapes (the accumulators take tensor-memory columns 0..255 either
// way, the converted-weight ring the other 256):
//   TOK = 256: 128 channels x 256 tokens, one M = 128, N = 256 MMA per K step
//              (an M = 128 MMA runs at the full rate only at N = 256);
//   TOK = 128: 256 channels x 128 tokens, two M = 128, N = 128 MMAs into two
//              accumulators, for small groups (less padding of the last tile).
// The epilogue applies s_x s_w and writes the transposed accumulators (TMEM
// lanes are channels), 32 channels of one token row a store.  Blockwise
// weight scales: each block scale is divided by the channel's largest one,
// S, and the quotient r, held as an f16 pair r_hi + r_lo (r to about 22
// bits), multiplies the block's converted codes in one fused f16
// multiply-add, q r_hi + (q r_lo), so each converted weight q r carries a
// single f16 rounding; S leaves the sum, and one accumulator runs over the
// whole K loop.
constexpr int kW8Ks = 64;                 // K per stage: 64 code bytes, one 128-byte f16 row
constexpr int kW8BoxBytes = 128 * kW8Ks;  // one u8 TMA box: 128 rows x 64 bytes (64-byte swizzle)
constexpr int kW8MaxRawStages = 6;
constexpr int kW8AColBase = 256;          // the converted-weight ring's first tensor-memory column
constexpr int kW8MaxAStages = 8, kW8MaxXStages = 4;
constexpr int kW8EpiWarps = 8;

struct W8Ctl {
  uint64_t rfull[kW8MaxRawStages];   // a stage's boxes have landed
  uint64_t rempty[kW8MaxRawStages];  // every reader of the stage is done with it
  uint64_t afull[kW8MaxAStages];  // converted weights are in tensor memory
  uint64_t aempty[kW8MaxAStages]; // the MMAs that read them completed
  uint64_t xfull[kW8MaxXStages];  // converted activations are in shared memory
  uint64_t xempty[kW8MaxXStages];
  uint64_t dfull, dempty;         // the accumulators hold a finished tile / have been read
  uint64_t drain;
  uint64_t never;  // test hook: a barrier that nothing arrives on
  uint32_t tmem_base;
  int abort_flag;
  int no_abort;
  int err;
  int total_tiles;
  int gstart[kMaxGroups + 1];
  int tile_prefix[kMaxGroups + 1];
  int gsize[kMaxGroups];
};

// XF16: the activations come as f16 codes from global memory (TMA, 128-byte
// swizzle, read by the MMA where they land) instead of e4m3 codes converted
// on the SM.
template <int TOK, bool XF16>
struct W8Cfg {
  static_assert(TOK == 128 || TOK == 256, "int8-weight tile: 128 or 256 tokens");
  static constexpr int HALVES = TOK == 128 ? 2 : 1;  // 128-channel weight tiles (MMA A operands) per tile
  static constexpr int CH = 128 * HALVES;             // channels per tile
  static constexpr int XBOXES = TOK / 128;            // activation boxes (128 rows) per stage
  static constexpr int XBOX_BYTES = XF16 ? 128 * kW8Ks * 2 : kW8BoxBytes;
  static constexpr int RAW_BYTES = HALVES * kW8BoxBytes + XBOXES * XBOX_BYTES;
  static constexpr int RAW_STAGES = RAW_BYTES > 3 * kW8BoxBytes ? 5 : 6;
  // weight converter warps: four per 128 channels; with XF16 and one weight
  // tile, two sets of four that take alternate stages (so that a stage's
  // conversion overlaps the next one's)
  static constexpr int WSETS = (XF16 && HALVES == 1) ? 2 : 1;
  static constexpr int WCONV = 4 * HALVES * WSETS;
  static constexpr int XCONV = XF16 ? 0 : TOK / 32;   // activation converter warps
  static constexpr int CONV = WCONV + XCONV;
  // readers of a raw stage: the converter warps, and with XF16 the MMAs (one commit)
  static constexpr int RAW_READERS = CONV / WSETS + (XF16 ? 1 : 0);
  static constexpr int XSTAGES = XF16 ? 0 : (TOK == 128 ? 4 : 2);  // ring of converted activation tiles
  static constexpr int XBYTES = TOK * kW8Ks * 2;
  static constexpr int ACOLS = 32 * HALVES;           // tensor-memory columns of one converted-weight stage
  static constexpr int ASTAGES = (512 - kW8AColBase) / ACOLS;
  static constexpr uint32_t IDESC = idesc_f16_f32(128, TOK);
  // warp 0 TMA producer, 1 MMA issuer, then the weight converters, the
  // activation converters and the 8 epilogue warps
  static constexpr int WARPS = 2 + CONV + kW8EpiWarps;
  static constexpr size_t SMEM = 1024 + static_cast<size_t>(RAW_STAGES) * RAW_BYTES +
                                 static_cast<size_t>(XSTAGES) * XBYTES + sizeof(W8Ctl);
  static_assert(XF16 || CONV == 12, "int8-weight roles");
  static_assert(RAW_STAGES <= kW8MaxRawStages && ASTAGES <= kW8MaxAStages && XSTAGES <= kW8MaxXStages &&
                    HALVES * TOK <= kW8AColBase && RAW_BYTES % 1024 == 0,
                "int8-weight buffer plan");
  static_assert(SMEM <= 232448, "int8-weight gmm: shared memory per CTA");
};

struct W8Tile {
  int el;    // local group
  int row0;  // first row (token) of the tile
  int rows;  // valid rows in the tile
  int n0;    // first channel
  int by;    // first weight row: el * N + n0
};

// Tile t: expert-major, then channel tile, then token tile (so that the CTAs
// running at the same time share one expert's weights), from the group
// tables built with units of TOK rows.
template <int TOK, int CH>
__device__ __forceinline__ W8Tile w8_tile(const Params& p, const W8Ctl* ctl, int t) {
  int lo = 0, hi = p.El;  // tile_prefix[lo] <= t < tile_prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (ctl->tile_prefix[mid] <= t) lo = mid; else hi = mid;
  }
  while (lo + 1 < p.El && ctl->tile_prefix[lo + 1] <= t) ++lo;  // skip empty groups
  const int sz = ctl->gsize[lo];
  const int mt = (sz + TOK - 1) / TOK;
  const int local = t - ctl->tile_prefix[lo];
  const int nt = local / mt, mi = local - nt * mt;
  W8Tile tl;
  tl.el = lo;
  tl.row0 = ctl->gstart[lo] + mi * TOK;
  tl.rows = min(TOK, sz - mi * TOK);
  tl.n0 = nt * CH;
  tl.by = lo * p.N + tl.n0;
  return tl;
}

// Blockwise weight scales of one channel: its largest block scale (0 for a
// channel past N).
__device__ __forceinline__ float w8_block_smax(const float* s_blk, int kblocks, int N, bool ok) {
  float m = 0.0f;
  if (ok)
    for (int kb = 0; kb < kblocks; ++kb) m = fmaxf(m, __ldg(s_blk + static_cast<int64_t>(kb) * N));
  return m;
}

template <int TOK, bool XF16>
__global__ void __launch_bounds__(W8Cfg<TOK, XF16>::WARPS * 32, 1)
    w8_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, const Params p) {
  using C = W8Cfg<TOK, XF16>;
  constexpr int NRAW = C::RAW_STAGES, RAWB = C::RAW_BYTES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  const uint32_t xring = base + NRAW * RAWB;  // converted activation tiles (without XF16)
  W8Ctl* ctl = reinterpret_cast<W8Ctl*>(base_ptr + NRAW * RAWB + C::XSTAGES * C::XBYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // group tables in units of TOK rows (two 128-row M tiles a unit for TOK = 256)
  if (warp == 0) build_group_tables<false, TOK == 256>(p, ctl);
  if (threadIdx.x == 32) {
    for (int s = 0; s < NRAW; ++s) {
      mbar_init(smem_u32(&ctl->rfull[s]), 1);
      mbar_init(smem_u32(&ctl->rempty[s]), C::RAW_READERS);
    }
    for (int a = 0; a < C::ASTAGES; ++a) {
      mbar_init(smem_u32(&ctl->afull[a]), C::WCONV / C::WSETS);
      mbar_init(smem_u32(&ctl->aempty[a]), 1);
    }
    for (int x = 0; x < C::XSTAGES; ++x) {
      mbar_init(smem_u32(&ctl->xfull[x]), C::XCONV);
      mbar_init(smem_u32(&ctl->xempty[x]), 1);
    }
    mbar_init(smem_u32(&ctl->dfull), 1);
    mbar_init(smem_u32(&ctl->dempty), kW8EpiWarps);
    mbar_init(smem_u32(&ctl->drain), 1);
    mbar_init(smem_u32(&ctl->never), 1);
    ctl->abort_flag = 0;
    ctl->no_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (ctl->err) {
    if (threadIdx.x == 0) raise_error(&g_err, MOE_DEVERR_GROUP_SIZES);
    return;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  const int total = ctl->total_tiles;
  const int nks = (p.K + kW8Ks - 1) / kW8Ks;
  const bool w_blk = p.rhs_mode == MOE_SCALE_PER_ROW_BLOCK128;
  volatile int* abort_flag = &ctl->abort_flag;
  bool timed_out = false;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = 0;
      for (int t = blockIdx.x; t < total && !timed_out; t += gridDim.x) {
        const W8Tile tl = w8_tile<TOK, C::CH>(p, ctl, t);
        for (int ks = 0; ks < nks; ++ks) {
          const int s = it % NRAW;
          if (!mbar_wait_bounded(smem_u32(&ctl->rempty[s]), ((it / NRAW) & 1) ^ 1, abort_flag, kWaitLimitNs)) {
            timed_out = true;
            break;
          }
          const uint32_t sa = base + s * RAWB, fb = smem_u32(&ctl->rfull[s]);
          mbar_arrive_expect_tx(fb, RAWB);
#pragma unroll
          for (int h = 0; h < C::HALVES; ++h)  // weight rows (channels) n0 + 128 h ..
            tma_load_2d(sa + h * kW8BoxBytes, &tmW, ks * kW8Ks, tl.by + 128 * h, fb);
#pragma unroll
          for (int b = 0; b < C::XBOXES; ++b)  // token rows row0 + 128 b .. (x: K elements either way)
            tma_load_2d(sa + C::HALVES * kW8BoxBytes + b * C::XBOX_BYTES, &tmX, ks * kW8Ks, tl.row0 + 128 * b, fb);
          ++it;
        }
      }
      if (timed_out) {
        *abort_flag = 1;
        ctl->err = 2;
        // let the loads already issued land before the CTA can exit
        for (uint32_t j = (it > NRAW ? it - NRAW : 0); j < it; ++j)
          mbar_wait_bounded(smem_u32(&ctl->rfull[j % NRAW]), (j / NRAW) & 1, &ctl->no_abort, kWaitLimitNs);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t it = 0, tcount = 0;
      for (int t = blockIdx.x; t < total && !timed_out; t += gridDim.x) {
        if (!mbar_wait_bounded(smem_u32(&ctl->dempty), (tcount & 1) ^ 1, abort_flag, kWaitLimitNs)) {
          timed_out = true;
          break;
        }
        tc_fence_after();
        for (int ks = 0; ks < nks; ++ks) {
          const int a = it % C::ASTAGES;
          // B: the converted tile (ring x) or, with XF16, the raw stage's f16 boxes
          const int x = XF16 ? static_cast<int>(it % NRAW) : static_cast<int>(it % (XF16 ? 1 : C::XSTAGES));
          const uint32_t bfull = XF16 ? smem_u32(&ctl->rfull[x]) : smem_u32(&ctl->xfull[x]);
          const uint32_t bpar = XF16 ? (it / NRAW) & 1 : (it / (XF16 ? 1 : C::XSTAGES)) & 1;
          if (!mbar_wait_bounded(smem_u32(&ctl->afull[a]), (it / C::ASTAGES) & 1, abort_flag, kWaitLimitNs) ||
              !mbar_wait_bounded(bfull, bpar, abort_flag, kWaitLimitNs)) {
            timed_out = true;
            break;
          }
          tc_fence_after();
          const uint64_t db = XF16 ? smem_desc_sw128(base + x * RAWB + C::HALVES * kW8BoxBytes)
                                   : smem_desc_sw128(xring + x * C::XBYTES);
          const uint32_t at = tmem_base + kW8AColBase + C::ACOLS * a;
#pragma unroll
          for (int h = 0; h < C::HALVES; ++h)
#pragma unroll
            for (int k16 = 0; k16 < kW8Ks / 16; ++k16)  // K = 16: 8 tensor-memory columns, 32 bytes of a B row
              mma_f16_tmem_a(tmem_base + TOK * h, at + 32 * h + 8 * k16, db + 2 * k16, C::IDESC,
                             (ks > 0 || k16 > 0) ? 1u : 0u);
          mma_commit(smem_u32(&ctl->aempty[a]));
          mma_commit(XF16 ? smem_u32(&ctl->rempty[x]) : smem_u32(&ctl->xempty[x]));
          ++it;
        }
        if (timed_out) break;
        mma_commit(smem_u32(&ctl->dfull));
        ++tcount;
      }
      // drain: every MMA this thread issued has completed once `drain` flips
      mma_commit(smem_u32(&ctl->drain));
      if (!mbar_wait_bounded(smem_u32(&ctl->drain), 0, &ctl->no_abort, kWaitLimitNs)) timed_out = true;
      if (timed_out) {
        *abort_flag = 1;
        ctl->err = 2;
      }
    }
    __syncwarp();
  } else if (warp < 2 + C::WCONV) {
    // --------------------------------------------------- weight converters
    // warp (h, q): rows 32 q .. 32 q + 31 of weight tile h (the tile's
    // channels 128 h ..), which are the tensor-memory lanes of that quarter;
    // with two sets, set `wset` takes the stages it with it % 2 == wset
    const int grp = (warp - 2) >> 2, q4 = warp & 3;
    const int h = grp % C::HALVES, wset = grp / C::HALVES;
    const int r = 32 * q4 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q4) << 16;
    const int swz = (r >> 1) & 3;  // 64-byte swizzle: 16-byte chunk j of row r sits at j ^ ((r / 2) % 4)
    uint32_t it = 0;
    for (int t = blockIdx.x; t < total && !timed_out; t += gridDim.x) {
      const W8Tile tl = w8_tile<TOK, C::CH>(p, ctl, t);
      const int ch = tl.n0 + 128 * h + r;
      const bool ch_ok = ch < p.N;
      const float* s_blk = p.rhs_scale + static_cast<int64_t>(tl.el) * p.kblocks * p.N + (ch_ok ? ch : 0);
      float inv_smax = 0.0f;
      if (w_blk) {
        const float m = w8_block_smax(s_blk, p.kblocks, p.N, ch_ok);
        inv_smax = m > 0.0f ? __frcp_rn(m) : 0.0f;
      }
      uint32_t rhi2 = 0x3C003C00u, rlo2 = 0u;  // f16x2 (1, 1) and (0, 0)
      int kb_have = -1;                        // the K block rhi2 / rlo2 belong to
      for (int ks = 0; ks < nks; ++ks) {
        if (C::WSETS > 1 && static_cast<int>(it % C::WSETS) != wset) {  // the other set's stage
          ++it;
          continue;
        }
        const int s = it % NRAW;
        if (!mbar_wait_bounded_warp(smem_u32(&ctl->rfull[s]), (it / NRAW) & 1, abort_flag, kWaitLimitNs)) {
          timed_out = true;
          break;
        }
        const uint8_t* src = base_ptr + s * RAWB + h * kW8BoxBytes + r * kW8Ks;
        uint4 wv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) wv[j] = *reinterpret_cast<const uint4*>(src + 16 * (j ^ swz));
        // the stage is refilled by TMA (the async proxy): order these generic
        // reads before that write, or the refill may land under them
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->rempty[s]));
        if (w_blk && (ks >> 1) != kb_have) {  // a new 128-wide K block (two stages)
          kb_have = ks >> 1;
          const float rel = ch_ok ? __fmul_rn(__ldg(s_blk + static_cast<int64_t>(kb_have) * p.N), inv_smax) : 0.0f;
          const __half hi = __float2half_rn(rel);
          const uint32_t hb = __half_as_ushort(hi);
          const uint32_t lb = __half_as_ushort(__float2half_rn(__fsub_rn(rel, __half2float(hi))));
          rhi2 = hb | (hb << 16);
          rlo2 = lb | (lb << 16);
        }
        const int a = it % C::ASTAGES;
        if (!mbar_wait_bounded_warp(smem_u32(&ctl->aempty[a]), ((it / C::ASTAGES) & 1) ^ 1, abort_flag,
                                    kWaitLimitNs)) {
          timed_out = true;
          break;
        }
        tc_fence_after();
        uint32_t f[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t wd[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            // bytes b0..b3 (K = 16 j + 4 c ..): b ^ 0x80 = b + 128 under the
            // f16 exponent of 1024 is 1152 + b exactly; minus 1152 leaves b
            const uint32_t x = wd[c] ^ 0x80808080u;
            uint32_t lo, hi;
            asm("prmt.b32 %0, %1, %2, 0x7170;" : "=r"(lo) : "r"(x), "r"(0x64646464u));
            asm("prmt.b32 %0, %1, %2, 0x7372;" : "=r"(hi) : "r"(x), "r"(0x64646464u));
            asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(0x64806480u));
            asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(0x64806480u));
            if (w_blk) {  // q r_hi + (q r_lo): one rounding of q r
              uint32_t t0, t1;
              asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(t0) : "r"(lo), "r"(rlo2));
              asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(t1) : "r"(hi), "r"(rlo2));
              asm("fma.rn.f16x2 %0, %0, %1, %2;" : "+r"(lo) : "r"(rhi2), "r"(t0));
              asm("fma.rn.f16x2 %0, %0, %1, %2;" : "+r"(hi) : "r"(rhi2), "r"(t1));
            }
            f[8 * j + 2 * c] = lo;      // K pair (16 j + 4 c, + 1): column 8 j + 2 c
            f[8 * j + 2 * c + 1] = hi;
          }
        }
        tmem_st_32x32b_x32(tmem_base + lane_addr + kW8AColBase + C::ACOLS * a + 32 * h, f);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->afull[a]));
        ++it;
      }
    }
    if (timed_out) {
      *abort_flag = 1;
      ctl->err = 2;
    }
  } else if (!XF16 && warp < 2 + C::CONV) {
    // ----------------------------------------------- activation converters
    const int r = 32 * (warp - 2 - C::WCONV) + lane;  // token row of the tile
    const int swz = (r >> 1) & 3;                      // the same within its 128-row box
    uint32_t it = 0;
    for (int t = blockIdx.x; t < total && !timed_out; t += gridDim.x) {
      for (int ks = 0; ks < nks; ++ks) {
        const int s = it % NRAW;
        if (!mbar_wait_bounded_warp(smem_u32(&ctl->rfull[s]), (it / NRAW) & 1, abort_flag, kWaitLimitNs)) {
          timed_out = true;
          break;
        }
        const uint8_t* src =
            base_ptr + s * RAWB + C::HALVES * kW8BoxBytes + (r >> 7) * C::XBOX_BYTES + (r & 127) * kW8Ks;
        uint4 xv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) xv[j] = *reinterpret_cast<const uint4*>(src + 16 * (j ^ swz));
        fence_proxy_async_smem();  // as above: generic reads before the TMA refill
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->rempty[s]));
        const int x = it % (XF16 ? 1 : C::XSTAGES);
        if (!mbar_wait_bounded_warp(smem_u32(&ctl->xempty[x]), ((it / (XF16 ? 1 : C::XSTAGES)) & 1) ^ 1, abort_flag,
                                    kWaitLimitNs)) {
          timed_out = true;
          break;
        }
        // row r of the f16 tile: 128 bytes in 8-row / 1024-byte atoms, its
        // 16-byte chunk c at c ^ (r % 8) (the 128-byte swizzle)
        uint8_t* dst = base_ptr + (xring - base) + x * C::XBYTES + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t wd[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
          uint32_t o[8];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint16_t lo16 = static_cast<uint16_t>(wd[c] & 0xFFFFu), hi16 = static_cast<uint16_t>(wd[c] >> 16);
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(o[2 * c]) : "h"(lo16));
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(o[2 * c + 1]) : "h"(hi16));
          }
          *reinterpret_cast<uint4*>(dst + 16 * ((2 * j) ^ (r & 7))) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(dst + 16 * ((2 * j + 1) ^ (r & 7))) = make_uint4(o[4], o[5], o[6], o[7]);
        }
        fence_proxy_async_smem();  // the tensor core reads the tile through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->xfull[x]));
        ++it;
      }
    }
    if (timed_out) {
      *abort_flag = 1;
      ctl->err = 2;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // warp (g, q): accumulator columns 128 g .. 128 g + 127 in lane quarter
    // q; with TOK = 128 those are all 128 tokens of channel half g, with
    // TOK = 256 tokens 128 g .. of the tile's 128 channels
    const int g = (warp - 2 - C::CONV) >> 2, q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const int ch_off = TOK == 128 ? 128 * g : 0, tok0 = TOK == 128 ? 0 : 128 * g;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q4) << 16;
    uint16_t* out = static_cast<uint16_t*>(p.out);
    uint32_t tcount = 0;
    if (p.stall && !mbar_wait_bounded_warp(smem_u32(&ctl->never), 0, abort_flag, p.stall_ns)) timed_out = true;
    for (int t = blockIdx.x; t < total && !timed_out; t += gridDim.x) {
      const W8Tile tl = w8_tile<TOK, C::CH>(p, ctl, t);
      const int ch = tl.n0 + ch_off + r;
      const bool ch_ok = ch < p.N;
      float s_w;
      if (w_blk)
        s_w = w8_block_smax(p.rhs_scale + static_cast<int64_t>(tl.el) * p.kblocks * p.N + (ch_ok ? ch : 0),
                            p.kblocks, p.N, ch_ok);
      else if (p.rhs_mode == MOE_SCALE_PER_ROW)
        s_w = ch_ok ? __ldg(p.rhs_scale + static_cast<int64_t>(tl.el) * p.N + ch) : 0.0f;
      else
        s_w = __ldg(p.rhs_scale);
      // token scales: lane j holds those of the warp's tokens j, 32 + j, 64 + j, 96 + j
      float sx[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int tok = tok0 + 32 * c + lane;
        sx[c] = p.lhs_mode == MOE_SCALE_PER_ROW ? (tok < tl.rows ? __ldg(p.lhs_scale + tl.row0 + tok) : 0.0f)
                                                : __ldg(p.lhs_scale);
      }
      if (!mbar_wait_bounded_warp(smem_u32(&ctl->dfull), tcount & 1, abort_flag, kWaitLimitNs)) {
        timed_out = true;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_base + lane_addr + 128 * g + 32 * c, v);
        tmem_wait_ld();
        if (c == 3) {  // the accumulators are read: the next tile's MMAs may start
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ctl->dempty));
        }
        uint16_t* orow = out + (static_cast<int64_t>(tl.row0) + tok0 + 32 * c) * p.N + ch;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float sxj = __shfl_sync(0xffffffffu, sx[c], j);
          if (ch_ok && tok0 + 32 * c + j < tl.rows)
            orow[static_cast<int64_t>(j) * p.N] =
                static_cast<uint16_t>(pack_bf16x2(__fmul_rn(__uint_as_float(v[j]), __fmul_rn(s_w, sxj)), 0.0f));
        }
      }
      ++tcount;
    }
    if (timed_out) {
      *abort_flag = 1;
      ctl->err = 2;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
  if (threadIdx.x == 0 && ctl->err) raise_error(&g_err, MOE_DEVERR_TIMEOUT);
}

// ---- helpers for the padded / sharded layouts ----------------------------

// Global first row of every group [0, E] into shared memory (warp 0).
__device__ void group_starts_smem(const int32_t* sizes, int E, int* starts) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    for (int c = 0; c < E; c += 32) {
      const int g = c + lane;
      const int v = g < E ? __ldg(sizes + g) : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (g < E) starts[g] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) starts[E] = carry;
  }
  __syncthreads();
}

// Zero the rows of a gmm output that lie outside groups [g0, g0 + El).
__global__ void zero_outside_kernel(uint16_t* out, int64_t M, int64_t N, const int32_t* sizes, int E, int g0,
                                    int El) {
  __shared__ int starts[kMaxGroups + 1];
  group_starts_smem(sizes, E, starts);
  const int64_t lo = starts[g0], hi = starts[g0 + El];
  const int64_t nvec = N / 8;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < M * nvec;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = i / nvec;
    if (row < lo || row >= hi) reinterpret_cast<uint4*>(out)[i] = make_uint4(0, 0, 0, 0);
  }
}

// e4m3 codes -> their f16 values (exact: f16 holds every e4m3 value), 16
// codes a thread and step: the int8-weight gmm's activations in the form its
// MMA reads.
__global__ void __launch_bounds__(256) e4m3_to_f16_kernel(const uint8_t* src, int64_t n16, uint16_t* dst) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint16_t lo16 = static_cast<uint16_t>(w[c] & 0xFFFFu), hi16 = static_cast<uint16_t>(w[c] >> 16);
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(o[2 * c]) : "h"(lo16));
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(o[2 * c + 1]) : "h"(hi16));
    }
    uint4* d = reinterpret_cast<uint4*>(dst) + 2 * i;
    d[0] = make_uint4(o[0], o[1], o[2], o[3]);
    d[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// src [M, C] e4m3 -> dst [C, Mp]: local group el's rows land at columns
// [pst(el), pst(el) + size), zero-filled up to the next multiple of 128.
// Persistent CTAs build the group tables once and walk 128 x 128 byte tiles
// (column tiles fastest).  A tile comes in with four 16-byte loads per thread
// (each source row segment read whole by eight lanes; the next tile's loads
// are issued before the current one is written out) and is staged in shared
// memory with its 16-byte units XOR-swizzled by 16-row group, so that both
// the stores and the transposing reads are free of bank conflicts.  Each
// thread then reads a 16-row x 4-byte strip as sixteen words, transposes its
// 4 x 4 byte blocks with byte permutes, and writes four 16-byte pieces; eight
// consecutive lanes cover one 128-byte run of an output row.
constexpr int kTpTile = 128;
__global__ void __launch_bounds__(256) transpose_pad_kernel(const uint8_t* src, int64_t M, int64_t C, uint8_t* dst,
                                                            int64_t Mp, const int32_t* sizes, int E, int g0,
                                                            int El) {
  __shared__ int starts[kMaxGroups + 1];
  __shared__ int pst[kMaxGroups + 1];
  __shared__ __align__(16) uint32_t tile[2][kTpTile][kTpTile / 4];
  group_starts_smem(sizes, E, starts);
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    for (int c = 0; c < El; c += 32) {
      const int el = c + lane;
      const int sz = el < El ? starts[g0 + el + 1] - starts[g0 + el] : 0;
      const int v = ((sz + 127) / 128) * 128;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (el < El) pst[el] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) pst[El] = carry;
  }
  __syncthreads();
  const int64_t rows_out = min(static_cast<int64_t>(pst[El]), Mp);  // padded columns of dst (a multiple of 128)
  const int64_t ntc = (C + kTpTile - 1) / kTpTile;
  const int64_t ntiles = (rows_out / kTpTile) * ntc;
  const int tid = threadIdx.x;
  const int lrow = tid >> 3, unit = tid & 7;  // load: rows lrow + 32 i, 16-byte unit `unit`
  auto load = [&](int64_t t, uint4 (&v)[4]) {
    const int64_t jb = (t / ntc) * kTpTile, cb = (t % ntc) * kTpTile;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t j = jb + lrow + 32 * i;
      const int64_t c = cb + 16 * unit;
      v[i] = make_uint4(0, 0, 0, 0);
      if (c < C) {
        int lo = 0, hi = El;
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (pst[mid] <= j) lo = mid; else hi = mid;
        }
        while (lo + 1 < El && pst[lo + 1] <= j) ++lo;
        const int64_t off = j - pst[lo];
        const int64_t sz = starts[g0 + lo + 1] - starts[g0 + lo];
        if (off < sz) {
          const int64_t m = starts[g0 + lo] + off;
          if (m < M) v[i] = __ldg(reinterpret_cast<const uint4*>(src + m * C + c));
        }
      }
    }
  };
  int64_t t = blockIdx.x;
  uint4 nxt[4];
  if (t < ntiles) load(t, nxt);
  const int rg = tid & 7, cw = tid >> 3;  // transpose: source rows 16 rg .. + 15, output rows 4 cw .. 4 cw + 3
  for (int b = 0; t < ntiles; t += gridDim.x, b ^= 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = lrow + 32 * i;
      *reinterpret_cast<uint4*>(&tile[b][r][4 * (unit ^ ((r >> 4) & 7))]) = nxt[i];
    }
    if (t + gridDim.x < ntiles) load(t + gridDim.x, nxt);
    __syncthreads();  // the two buffers alternate, so one barrier per tile suffices
    const int64_t jb = (t / ntc) * kTpTile, cb = (t % ntc) * kTpTile;
    const int wsw = (cw & 3) | (((cw >> 2) ^ rg) << 2);  // word column cw after the swizzle of group rg
    uint32_t o[4][4];  // o[k][q]: output row 4 cw + k, source rows 16 rg + 4 q .. + 3
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = 16 * rg + 4 * q;
      const uint32_t r0 = tile[b][r][wsw], r1 = tile[b][r + 1][wsw];
      const uint32_t r2 = tile[b][r + 2][wsw], r3 = tile[b][r + 3][wsw];
      const uint32_t t0 = __byte_perm(r0, r1, 0x5140), t1 = __byte_perm(r2, r3, 0x5140);
      const uint32_t t2 = __byte_perm(r0, r1, 0x7362), t3 = __byte_perm(r2, r3, 0x7362);
      o[0][q] = __byte_perm(t0, t1, 0x5410);
      o[1][q] = __byte_perm(t0, t1, 0x7632);
      o[2][q] = __byte_perm(t2, t3, 0x5410);
      o[3][q] = __byte_perm(t2, t3, 0x7632);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t c = cb + 4 * cw + k;
      if (c < C)
        *reinterpret_cast<uint4*>(dst + c * Mp + jb + 16 * rg) = make_uint4(o[k][0], o[k][1], o[k][2], o[k][3]);
    }
  }
}

// g bf16 [M, C] -> dst [C, Mp]: the per-(group, column) e4m3 codes of g
// (finished scales `scale` [El, C]) written straight into the transposed,
// group-padded layout that the tgmm contraction reads; the same tiles,
// swizzle and byte-permute transpose as transpose_pad_kernel, with the
// quantisation of moe_quantize_group_cols in between (bit-identical codes).
// A 128-row tile of the padded layout lies inside one group, so a thread's
// eight column scales are loaded once per tile.
__global__ void __launch_bounds__(256) quant_transpose_pad_kernel(const uint16_t* g, int64_t M, int64_t C,
                                                                  const float* scale, uint8_t* dst, int64_t Mp,
                                                                  const int32_t* sizes, int E, int g0, int El) {
  __shared__ int starts[kMaxGroups + 1];
  __shared__ int pst[kMaxGroups + 1];
  __shared__ __align__(16) uint32_t tile[kTpTile][kTpTile / 4];
  group_starts_smem(sizes, E, starts);
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    for (int c = 0; c < El; c += 32) {
      const int el = c + lane;
      const int sz = el < El ? starts[g0 + el + 1] - starts[g0 + el] : 0;
      const int v = ((sz + 127) / 128) * 128;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (el < El) pst[el] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) pst[El] = carry;
  }
  __syncthreads();
  const int64_t rows_out = min(static_cast<int64_t>(pst[El]), Mp);
  const int64_t ntc = (C + kTpTile - 1) / kTpTile;
  const int64_t ntiles = (rows_out / kTpTile) * ntc;
  const int tid = threadIdx.x;
  const int lrow = tid >> 4, unit = tid & 15;  // load: rows lrow + 16 i, 8 columns 8 unit .. 8 unit + 7
  const int rg = tid & 7, cw = tid >> 3;       // transpose: as transpose_pad_kernel
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int64_t jb = (t / ntc) * kTpTile, cb = (t % ntc) * kTpTile;
    // the tile's group (every row of a 128-row padded tile belongs to it)
    int lo = 0, hi = El;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pst[mid] <= jb) lo = mid; else hi = mid;
    }
    while (lo + 1 < El && pst[lo + 1] <= jb) ++lo;
    const int64_t sz = starts[g0 + lo + 1] - starts[g0 + lo];
    const int64_t c0 = cb + 8 * unit;
    float sc[8], inv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      sc[j] = (c0 + j < C) ? __ldg(scale + static_cast<int64_t>(lo) * C + c0 + j) : 1.0f;
      inv[j] = __frcp_rn(sc[j]);
    }
    uint4 d[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t off = jb + lrow + 16 * i - pst[lo];
      d[i] = make_uint4(0, 0, 0, 0);
      if (off < sz && c0 < C) {
        const int64_t m = starts[g0 + lo] + off;
        if (m < M) d[i] = __ldg(reinterpret_cast<const uint4*>(g + m * C + c0));
      }
    }
    __syncthreads();  // the previous tile's transposing reads are done
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = lrow + 16 * i;
      const uint32_t w[4] = {d[i].x, d[i].y, d[i].z, d[i].w};
      float v[8], y[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[2 * j] = bf16lo(w[j]);
        v[2 * j + 1] = bf16hi(w[j]);
      }
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
      const uint2 code = pack_e4m3x8(y);  // zero rows (padding) give zero codes
      // 8 bytes: half of 16-byte unit (unit >> 1), swizzled by 16-row group
      *reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(&tile[r][0]) + 16 * ((unit >> 1) ^ ((r >> 4) & 7)) +
                                8 * (unit & 1)) = code;
    }
    __syncthreads();
    const int wsw = (cw & 3) | (((cw >> 2) ^ rg) << 2);
    uint32_t o[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = 16 * rg + 4 * q;
      const uint32_t r0 = tile[r][wsw], r1 = tile[r + 1][wsw], r2 = tile[r + 2][wsw], r3 = tile[r + 3][wsw];
      const uint32_t t0 = __byte_perm(r0, r1, 0x5140), t1 = __byte_perm(r2, r3, 0x5140);
      const uint32_t t2 = __byte_perm(r0, r1, 0x7362), t3 = __byte_perm(r2, r3, 0x7362);
      o[0][q] = __byte_perm(t0, t1, 0x5410);
      o[1][q] = __byte_perm(t0, t1, 0x7632);
      o[2][q] = __byte_perm(t2, t3, 0x5410);
      o[3][q] = __byte_perm(t2, t3, 0x7632);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t c = cb + 4 * cw + k;
      if (c < C)
        *reinterpret_cast<uint4*>(dst + c * Mp + jb + 16 * rg) = make_uint4(o[k][0], o[k][1], o[k][2], o[k][3]);
    }
  }
}

// ---- fused SwiGLU: rows outside the local groups, per-row second phase ----

// Rows outside groups [g0, g0 + El) of a fused SwiGLU call get zero codes and
// scale 1, as the unfused path gives for its zero rows.  In the per-row mode
// their running maximum is set to -1 so that the code pass skips them and
// writes scale 1.
__global__ void swiglu_outside_kernel(uint8_t* h_q, float* h_scale, uint8_t* h_sf, int64_t M, int64_t F, int h_mode,
                                      const int32_t* sizes, int E, int g0, int El) {
  __shared__ int starts[kMaxGroups + 1];
  group_starts_smem(sizes, E, starts);
  const int64_t lo = starts[g0], hi = starts[g0 + El];
  const int64_t nvec = F / 16, nb = F / 128;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < M * nvec; i += stride) {
    const int64_t row = i / nvec;
    if (row < lo || row >= hi) reinterpret_cast<uint4*>(h_q)[i] = make_uint4(0, 0, 0, 0);
  }
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; row < M; row += stride) {
    if (row >= lo && row < hi) continue;
    if (h_mode == MOE_SCALE_PER_ROW) {
      h_scale[row] = -1.0f;
    } else if (h_mode == MOE_SCALE_PER_ROW_BLOCK128) {
      for (int64_t b = 0; b < nb; ++b) h_scale[row * nb + b] = 1.0f;
    } else if (h_sf) {  // MXFP8 (K-block-major words): a zero block's E8M0 code is 0
      for (int64_t b = 0; b < F / 128; ++b) reinterpret_cast<uint32_t*>(h_sf)[b * M + row] = 0;
    }
  }
}

// Second phase of the per-token h scales: the codes of one row against its
// finished amax (one CTA per row; a thread takes V pairs of adjacent 16-byte
// vectors, 16 columns each, all loads issued before any is used and before
// the row's amax is read, and writes each pair's codes with one 16-byte
// store), and the row's final scale amax / 448 written over the amax (1 for a
// row outside the local groups, whose amax slot holds a negative mark).
template <int V>
__global__ void __launch_bounds__(256) h_quant_rows_kernel(const uint16_t* h, float* h_scale, int npair, uint8_t* q) {
  const int64_t row = blockIdx.x;
  const uint4* hr = reinterpret_cast<const uint4*>(h) + row * 2 * npair;
  uint4* qr = reinterpret_cast<uint4*>(q) + row * npair;
  float m = 0.0f, s = 1.0f, inv = 1.0f;
  for (int base = 0; base < npair; base += V * blockDim.x) {
    uint4 d[V][2];
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int v = base + i * blockDim.x + threadIdx.x;
      if (v < npair) {
        d[i][0] = __ldg(hr + 2 * v);
        d[i][1] = __ldg(hr + 2 * v + 1);
      }
    }
    if (base == 0) {
      m = h_scale[row];
      s = absmax_scale(m);  // 1 for a negative mark
      inv = __frcp_rn(s);
      __syncthreads();  // every thread has read the amax before it is replaced
      if (threadIdx.x == 0) h_scale[row] = s;
    }
    if (m < 0.0f) return;  // outside the local groups
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int v = base + i * blockDim.x + threadIdx.x;
      if (v < npair) {
        uint2 c[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint32_t w[4] = {d[i][hh].x, d[i][hh].y, d[i][hh].z, d[i][hh].w};
          float x8[8], qv[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            x8[2 * j] = bf16lo(w[j]);
            x8[2 * j + 1] = bf16hi(w[j]);
          }
          quant_n<8>(x8, s, inv, qv);
          c[hh] = pack_e4m3x8(qv);
        }
        qr[v] = make_uint4(c[0].x, c[0].y, c[1].x, c[1].y);
      }
    }
  }
}


// ---- host side -----------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D uint8 tensor map: rows x inner bytes, box rows_box x 128, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint64_t pitch, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {pitch};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D uint8 tensor map for the int8-weight gmm: box rows_box x 64 bytes,
// 64-byte swizzle (16-byte chunk j of box row r at j ^ ((r / 2) % 4)); reads
// past the extents return zeros.
bool make_map_u8_64(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint64_t pitch,
                    uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {pitch};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kW8Ks), box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D bf16 tensor map: rows x inner elements (row pitch in bytes, a multiple
// of 16), box rows_box x 64 elements (128 bytes), 128-byte swizzle; reads past
// the extents return zeros.
bool make_map_bf16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint64_t pitch_bytes,
                   uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D fp32 tensor map of the tgmm output [E_local, K, N] for 32 x 32 stores
// with the 128-byte swizzle (rows >= K or columns >= N are clipped).
bool make_map_out_f32(CUtensorMap* m, void* ptr, uint64_t N, uint64_t K, uint64_t El) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {N, K, El};
  cuuint64_t strides[2] = {N * 4, K * N * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

bool device_is_sm103() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  return major == 10 && minor == 3;
}

// Units of work for a gmm launch: M tiles (pairs of M tiles on CTA pairs)
// times N tiles, bounded by the ragged-group worst case.
template <int MODE, bool PAIR_REQ>
int gmm_max_units(int64_t M, int E_local, int ntiles) {
  const int64_t rows_per_unit = (Cfg<MODE, PAIR_REQ>::PAIR ? 2 : 1) * BM;
  const int64_t u = ((M + rows_per_unit - 1) / rows_per_unit + E_local) * ntiles;
  return static_cast<int>(u > (1 << 30) ? (1 << 30) : u);
}

template <int MODE, bool PAIR_REQ>
moe_status launch_mma(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& O, const Params& p,
                      int max_units, cudaStream_t st) {
  using C = Cfg<MODE, PAIR_REQ>;
  auto kernel = mma_kernel<MODE, PAIR_REQ>;
  MOE_CUDA_TRY(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(C::SMEM)));
  if (C::SPLIT) {
    // the register split may only hand out what the CTA is launched with
    cudaFuncAttributes fa{};
    MOE_CUDA_TRY(cudaFuncGetAttributes(&fa, kernel));
    if (static_cast<int64_t>(fa.numRegs) * C::THREADS <
        128ll * C::CTRL_REGS + 32ll * C::EPI_WARPS * C::EPI_REGS)
      return MOE_ERR_UNSUPPORTED;
  }
  const int sms = sm_count();
  if (sms <= 0) return MOE_ERR_CUDA;
  if (max_units <= 0) max_units = 1;
  if (!C::PAIR) {
    const int grid = max_units < sms ? max_units : sms;
    kernel<<<grid, C::THREADS, C::SMEM, st>>>(A, B, O, p);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
  }
  // persistent CTA pairs: as many 2-CTA clusters as fit at once
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // resident clusters of this instantiation, cached per device (several
  // host threads may launch on several devices)
  static std::mutex mu;
  static int max_clusters[kMaxDevices] = {};
  int dev = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  int mc = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    mc = max_clusters[dev];
  }
  if (mc == 0) {
    cfg.gridDim = dim3(2 * (sms / 2));
    int n = 0;
    MOE_CUDA_TRY(cudaOccupancyMaxActiveClusters(&n, kernel, &cfg));
    if (n <= 0) return MOE_ERR_UNSUPPORTED;
    mc = n;
    std::lock_guard<std::mutex> lock(mu);
    max_clusters[dev] = n;
  }
  const int clusters = max_units < mc ? max_units : mc;
  cfg.gridDim = dim3(2 * clusters);
  MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, kernel, A, B, O, p));
  return MOE_OK;
}

// test hook (moe_test_stall_epilogue): 0, or the wait limit in ns
std::atomic<uint64_t> g_stall_ns{0};

// gmm_fp8_w8 with tiles of TOK tokens: one persistent CTA per SM at most.
template <int TOK, bool XF16>
moe_status launch_w8(const CUtensorMap& X, const CUtensorMap& W, Params p, int E_local, cudaStream_t st) {
  using C = W8Cfg<TOK, XF16>;
  p.ntiles = static_cast<int>((p.N + C::CH - 1) / C::CH);
  MOE_CUDA_TRY(cudaFuncSetAttribute(w8_kernel<TOK, XF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(C::SMEM)));
  const int sms = sm_count();
  if (sms <= 0) return MOE_ERR_CUDA;
  const int64_t units = ((p.M + TOK - 1) / TOK + E_local) * static_cast<int64_t>(p.ntiles);
  const int grid = units < sms ? static_cast<int>(units) : sms;
  w8_kernel<TOK, XF16><<<grid, C::WARPS * 32, C::SMEM, st>>>(X, W, p);
  MOE_CUDA_TRY(cudaGetLastError());
  return MOE_OK;
}

bool valid_lhs_mode(int m) {
  return m == MOE_SCALE_PER_ROW || m == MOE_SCALE_PER_ROW_BLOCK128 || m == MOE_SCALE_PER_TENSOR;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" __attribute__((visibility("hidden"))) cudaError_t moe_detail_take_error_gmm(unsigned int* out) {
  unsigned int v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_err, sizeof(v));
  if (e == cudaSuccess && v) e = cudaMemcpyToSymbol(g_err, &z, sizeof(z));
  *out = v;
  return e;
}

extern "C" int moe_num_sms(void) { return sm_count(); }

extern "C" void moe_test_stall_epilogue(uint64_t limit_ns) { g_stall_ns.store(limit_ns); }

extern "C" moe_status gmm_fp8(const uint8_t* lhs_q, const float* lhs_scale, moe_scale_mode lhs_mode,
                              const uint8_t* rhs_q, const float* rhs_scale, moe_scale_mode rhs_mode,
                              const int32_t* group_sizes, int E, int group_offset, int E_local, int64_t M, int64_t K,
                              int64_t N, uint16_t* out, moe_stream_t stream) {
  MOE_HOST_CHECK(lhs_q && lhs_scale && rhs_q && rhs_scale && group_sizes && out, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(valid_lhs_mode(lhs_mode) && valid_lhs_mode(rhs_mode), MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(E > 0 && E <= kMaxGroups && group_offset >= 0 && E_local > 0 && group_offset + E_local <= E,
                 MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(M >= 0 && M < (1ll << 31) && K > 0 && K % 16 == 0 && K < (1 << 30) && N > 0 && N % 16 == 0,
                 MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(static_cast<int64_t>(E_local) * N < (1ll << 31), MOE_ERR_INVALID_ARG);
  const bool blockwise = lhs_mode == MOE_SCALE_PER_ROW_BLOCK128 || rhs_mode == MOE_SCALE_PER_ROW_BLOCK128;
  MOE_HOST_CHECK(!blockwise || K % 128 == 0, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(aligned16(lhs_q) && aligned16(rhs_q) && aligned16(out), MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(rhs_mode == MOE_SCALE_PER_TENSOR || aligned16(rhs_scale), MOE_ERR_INVALID_ARG);
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  if (M == 0) return MOE_OK;
  if (group_offset > 0 || E_local < E) {
    zero_outside_kernel<<<sm_count() * 4, 256, 0, st>>>(out, M, N, group_sizes, E, group_offset, E_local);
    MOE_CUDA_TRY(cudaGetLastError());
  }
  CUtensorMap A, B;
  if (!make_map(&A, lhs_q, K, M, K, BM)) return MOE_ERR_CUDA;
  // CTA pairs pay off once the K loop is long enough to amortise the pair's
  // coupling (measured: slower at K <= 2048, 7-9% faster at K = 4096, 14336)
  const bool pair = !blockwise && Cfg<kFinal, true>::PAIR && K >= kPairMinK;
  const int bn = blockwise ? Cfg<kPromote>::BN : Cfg<kFinal>::BN;
  // B box: one tile of N rows, or this CTA's half of it on a CTA pair
  const uint32_t b_box = pair ? bn / 2 : bn;
  if (!make_map(&B, rhs_q, K, static_cast<uint64_t>(E_local) * N, K, b_box)) return MOE_ERR_CUDA;
  Params p{};
  p.group_sizes = group_sizes;
  p.E = E;
  p.g0 = group_offset;
  p.El = E_local;
  p.M = M;
  p.K = static_cast<int>(K);
  p.N = static_cast<int>(N);
  p.kblocks = static_cast<int>((K + BK - 1) / BK);
  p.ntiles = static_cast<int>((N + bn - 1) / bn);
  p.ktiles = 0;
  p.lhs_scale = lhs_scale;
  p.lhs_mode = lhs_mode;
  p.rhs_scale = rhs_scale;
  p.rhs_mode = rhs_mode;
  p.out = out;
  p.stall_ns = g_stall_ns.load();
  p.stall = p.stall_ns != 0;
  if (blockwise) return launch_mma<kPromote, false>(A, B, A, p, gmm_max_units<kPromote, false>(M, E_local, p.ntiles), st);
  if (pair) return launch_mma<kFinal, true>(A, B, A, p, gmm_max_units<kFinal, true>(M, E_local, p.ntiles), st);
  return launch_mma<kFinal, false>(A, B, A, p, gmm_max_units<kFinal, false>(M, E_local, p.ntiles), st);
}

extern "C" moe_status gmm_fp8_ksplit(const uint8_t* lhs_q, const float* lhs_scale, moe_scale_mode lhs_mode,
                                     const uint8_t* rhs_q, const float* rhs_scale2, int64_t K_split,
                                     const int32_t* group_sizes, int E, int group_offset, int E_local, int64_t M,
                                     int64_t K, int64_t N, uint16_t* out, moe_stream_t stream) {
  MOE_HOST_CHECK(lhs_q && lhs_scale && rhs_q && rhs_scale2 && group_sizes && out, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(lhs_mode == MOE_SCALE_PER_ROW || lhs_mode == MOE_SCALE_PER_TENSOR, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(E > 0 && E <= kMaxGroups && group_offset >= 0 && E_local > 0 && group_offset + E_local <= E,
                 MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(M >= 0 && M < (1ll << 31) && K > 0 && K % 16 == 0 && K < (1 << 30) && N > 0 && N % 16 == 0,
                 MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(K_split >= 0 && K_split <= K && K_split % BK == 0, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(static_cast<int64_t>(E_local) * N < (1ll << 31), MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(aligned16(lhs_q) && aligned16(rhs_q) && aligned16(out), MOE_ERR_INVALID_ARG);
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  if (M == 0) return MOE_OK;
  if (group_offset > 0 || E_local < E) {
    zero_outside_kernel<<<sm_count() * 4, 256, 0, st>>>(out, M, N, group_sizes, E, group_offset, E_local);
    MOE_CUDA_TRY(cudaGetLastError());
  }
  CUtensorMap A, B;
  if (!make_map(&A, lhs_q, K, M, K, BM)) return MOE_ERR_CUDA;
  if (!make_map(&B, rhs_q, K, static_cast<uint64_t>(E_local) * N, K, Cfg<kSplit>::BN)) return MOE_ERR_CUDA;
  Params p{};
  p.group_sizes = group_sizes;
  p.E = E;
  p.g0 = group_offset;
  p.El = E_local;
  p.M = M;
  p.K = static_cast<int>(K);
  p.N = static_cast<int>(N);
  p.kblocks = static_cast<int>((K + BK - 1) / BK);
  p.kb_split = static_cast<int>(K_split / BK);
  p.ntiles = static_cast<int>((N + Cfg<kSplit>::BN - 1) / Cfg<kSplit>::BN);
  p.ktiles = 0;
  p.lhs_scale = lhs_scale;
  p.lhs_mode = lhs_mode;
  p.rhs_scale = rhs_scale2;
  p.rhs_mode = MOE_SCALE_PER_TENSOR;
  p.out = out;
  return launch_mma<kSplit, false>(A, B, A, p, gmm_max_units<kSplit, false>(M, E_local, p.ntiles), st);
}

extern "C" moe_status gmm_fp8_swiglu(const uint8_t* lhs_q, const float* lhs_scale, moe_scale_mode lhs_mode,
                                     const uint8_t* rhs_q, const float* rhs_scale, moe_scale_mode rhs_mode,
                                     const int32_t* group_sizes, int E, int group_offset, int E_local, int64_t M,
                                     int64_t K, int64_t F, moe_scale_mode h_mode, const float* h_static_scale,
                                     uint16_t* a_out, uint16_t* h, uint8_t* h_q, float* h_scale,
                                     moe_stream_t stream) {
  MOE_HOST_CHECK(lhs_q && lhs_scale && rhs_q && rhs_scale && group_sizes && h_q, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(valid_lhs_mode(lhs_mode) && valid_lhs_mode(rhs_mode), MOE_ERR_INVALID_ARG);
  // a blockwise operand scale: the promotion kernel with the SwiGLU epilogue
  const bool blockwise = lhs_mode == MOE_SCALE_PER_ROW_BLOCK128 || rhs_mode == MOE_SCALE_PER_ROW_BLOCK128;
  MOE_HOST_CHECK(!blockwise || K % 128 == 0, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(E > 0 && E <= kMaxGroups && group_offset >= 0 && E_local > 0 && group_offset + E_local <= E,
                 MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(M >= 0 && M < (1ll << 31) && K > 0 && K % 16 == 0 && K < (1 << 30) && F > 0 && F % 128 == 0 &&
                     2 * static_cast<int64_t>(E_local) * F < (1ll << 31),
                 MOE_ERR_INVALID_ARG);
  if (h_mode == MOE_SCALE_PER_ROW) {
    MOE_HOST_CHECK(h && h_scale && aligned16(h), MOE_ERR_INVALID_ARG);
  } else if (h_mode == MOE_SCALE_PER_ROW_BLOCK128) {
    MOE_HOST_CHECK(h_scale != nullptr, MOE_ERR_INVALID_ARG);
  } else {
    MOE_HOST_CHECK(h_mode == MOE_SCALE_PER_TENSOR && h_static_scale, MOE_ERR_INVALID_ARG);
  }
  MOE_HOST_CHECK(aligned16(lhs_q) && aligned16(rhs_q) && aligned16(h_q) && (!a_out || aligned16(a_out)) &&
                     (rhs_mode == MOE_SCALE_PER_TENSOR || aligned16(rhs_scale)),
                 MOE_ERR_INVALID_ARG);
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  if (M == 0) return MOE_OK;
  if (h_mode == MOE_SCALE_PER_ROW) MOE_CUDA_TRY(cudaMemsetAsync(h_scale, 0, sizeof(float) * M, st));
  if (group_offset > 0 || E_local < E) {
    swiglu_outside_kernel<<<sm_count() * 4, 256, 0, st>>>(h_q, h_scale, nullptr, M, F, h_mode, group_sizes, E,
                                                            group_offset, E_local);
    MOE_CUDA_TRY(cudaGetLastError());
  }
  CUtensorMap A, B;
  if (!make_map(&A, lhs_q, K, M, K, BM)) return MOE_ERR_CUDA;
  if (!make_map(&B, rhs_q, K, static_cast<uint64_t>(E_local) * 2 * F, K, 128)) return MOE_ERR_CUDA;
  Params p{};
  p.group_sizes = group_sizes;
  p.E = E;
  p.g0 = group_offset;
  p.El = E_local;
  p.M = M;
  p.K = static_cast<int>(K);
  p.N = static_cast<int>(2 * F);
  p.kblocks = static_cast<int>((K + BK - 1) / BK);
  p.ntiles = static_cast<int>(F / 128);
  p.lhs_scale = lhs_scale;
  p.lhs_mode = lhs_mode;
  p.rhs_scale = rhs_scale;
  p.rhs_mode = rhs_mode;
  p.F = static_cast<int>(F);
  p.h_mode = h_mode;
  p.h_static = h_static_scale;
  p.a_out = a_out;
  p.h_out = h;
  p.h_q = h_q;
  p.h_scale = h_scale;
  moe_status stt =
      blockwise ? launch_mma<kPromoteSwiglu, false>(A, B, A, p, gmm_max_units<kPromoteSwiglu, false>(M, E_local, p.ntiles),
                                                    st)
      : K >= kPairMinK
          ? launch_mma<kSwiglu, true>(A, B, A, p, gmm_max_units<kSwiglu, true>(M, E_local, p.ntiles), st)
          : launch_mma<kSwiglu, false>(A, B, A, p, gmm_max_units<kSwiglu, false>(M, E_local, p.ntiles), st);
  if (stt != MOE_OK) return stt;
  if (h_mode == MOE_SCALE_PER_ROW) {
    const int npair = static_cast<int>(F / 16);  // F is a multiple of 128
    const int threads = std::min(256, ((npair + 4 * 32 - 1) / (4 * 32)) * 32);
    h_quant_rows_kernel<4><<<static_cast<unsigned>(M), threads, 0, st>>>(h, h_scale, npair, h_q);
    MOE_CUDA_TRY(cudaGetLastError());
  }
  return MOE_OK;
}

extern "C" moe_status gmm_fp8_mx(const uint8_t* lhs_q, const uint8_t* lhs_sf, const uint8_t* rhs_q,
                                 const uint8_t* rhs_sf, const int32_t* group_sizes, int E, int group_offset,
                                 int E_local, int64_t M, int64_t K, int64_t N, uint16_t* out, moe_stream_t stream) {
  MOE_HOST_CHECK(lhs_q && lhs_sf && rhs_q && rhs_sf && group_sizes && out, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(E > 0 && E <= kMaxGroups && group_offset >= 0 && E_local > 0 && group_offset + E_local <= E,
                 MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(M >= 0 && M < (1ll << 31) && K > 0 && K % 128 == 0 && K < (1 << 30) && N > 0 && N % 16 == 0,
                 MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(static_cast<int64_t>(E_local) * N < (1ll << 31), MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(aligned16(lhs_q) && aligned16(rhs_q) && aligned16(out) && aligned16(lhs_sf) && aligned16(rhs_sf),
                 MOE_ERR_INVALID_ARG);
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  if (M == 0) return MOE_OK;
  if (group_offset > 0 || E_local < E) {
    zero_outside_kernel<<<sm_count() * 4, 256, 0, st>>>(out, M, N, group_sizes, E, group_offset, E_local);
    MOE_CUDA_TRY(cudaGetLastError());
  }
  CUtensorMap A, B;
  if (!make_map(&A, lhs_q, K, M, K, BM)) return MOE_ERR_CUDA;
  if (!make_map(&B, rhs_q, K, static_cast<uint64_t>(E_local) * N, K, Cfg<kMx>::BN)) return MOE_ERR_CUDA;
  Params p{};
  p.group_sizes = group_sizes;
  p.E = E;
  p.g0 = group_offset;
  p.El = E_local;
  p.M = M;
  p.K = static_cast<int>(K);
  p.N = static_cast<int>(N);
  p.kblocks = static_cast<int>(K / BK);
  p.ntiles = static_cast<int>((N + Cfg<kMx>::BN - 1) / Cfg<kMx>::BN);
  p.lhs_sf = lhs_sf;
  p.rhs_sf = rhs_sf;
  p.out = out;
  p.stall_ns = g_stall_ns.load();
  p.stall = p.stall_ns != 0;
  return launch_mma<kMx, false>(A, B, A, p, gmm_max_units<kMx, false>(M, E_local, p.ntiles), st);
}

extern "C" moe_status gmm_fp8_mx_swiglu(const uint8_t* lhs_q, const uint8_t* lhs_sf, const uint8_t* rhs_q,
                                        const uint8_t* rhs_sf, const int32_t* group_sizes, int E, int group_offset,
                                        int E_local, int64_t M, int64_t K, int64_t F, uint16_t* a_out, uint8_t* h_q,
                                        uint8_t* h_sf, moe_stream_t stream) {
  MOE_HOST_CHECK(lhs_q && lhs_sf && rhs_q && rhs_sf && group_sizes && h_q && h_sf, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(E > 0 && E <= kMaxGroups && group_offset >= 0 && E_local > 0 && group_offset + E_local <= E,
                 MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(M >= 0 && M < (1ll << 31) && K > 0 && K % 128 == 0 && K < (1 << 30) && F > 0 && F % 128 == 0 &&
                     2 * static_cast<int64_t>(E_local) * F < (1ll << 31),
                 MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(aligned16(lhs_q) && aligned16(rhs_q) && aligned16(h_q) && aligned16(lhs_sf) && aligned16(rhs_sf) &&
                     (!a_out || aligned16(a_out)),
                 MOE_ERR_INVALID_ARG);
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  if (M == 0) return MOE_OK;
  if (group_offset > 0 || E_local < E) {
    swiglu_outside_kernel<<<sm_count() * 4, 256, 0, st>>>(h_q, nullptr, h_sf, M, F, -1, group_sizes, E, group_offset,
                                                            E_local);
    MOE_CUDA_TRY(cudaGetLastError());
  }
  CUtensorMap A, B;
  if (!make_map(&A, lhs_q, K, M, K, BM)) return MOE_ERR_CUDA;
  if (!make_map(&B, rhs_q, K, static_cast<uint64_t>(E_local) * 2 * F, K, 128)) return MOE_ERR_CUDA;
  Params p{};
  p.group_sizes = group_sizes;
  p.E = E;
  p.g0 = group_offset;
  p.El = E_local;
  p.M = M;
  p.K = static_cast<int>(K);
  p.N = static_cast<int>(2 * F);
  p.kblocks = static_cast<int>(K / BK);
  p.ntiles = static_cast<int>(F / 128);
  p.lhs_sf = lhs_sf;
  p.rhs_sf = rhs_sf;
  p.F = static_cast<int>(F);
  p.a_out = a_out;
  p.h_q = h_q;
  p.h_sf = h_sf;
  p.stall_ns = g_stall_ns.load();
  p.stall = p.stall_ns != 0;
  return launch_mma<kMxSwiglu, false>(A, B, A, p, gmm_max_units<kMxSwiglu, false>(M, E_local, p.ntiles), st);
}

namespace {
int64_t padded_rows(int64_t M, int E_local) { return ((M + 127) / 128) * 128 + 128ll * E_local; }
size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
}  // namespace

extern "C" size_t gmm_fp8_w8_workspace_bytes(int64_t M, int64_t K) {
  return (M > 0 && K > 0 && M < (1ll << 31) && K < (1 << 30)) ? static_cast<size_t>(2 * M * K) : 0;
}

extern "C" moe_status gmm_fp8_w8(const uint8_t* lhs_q, const float* lhs_scale, moe_scale_mode lhs_mode,
                                 const int8_t* rhs_q, const float* rhs_scale, moe_scale_mode rhs_mode,
                                 const int32_t* group_sizes, int E, int group_offset, int E_local, int64_t M,
                                 int64_t K, int64_t N, uint16_t* out, void* workspace, size_t workspace_bytes,
                                 moe_stream_t stream) {
  MOE_HOST_CHECK(lhs_q && lhs_scale && rhs_q && rhs_scale && group_sizes && out, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(lhs_mode == MOE_SCALE_PER_ROW || lhs_mode == MOE_SCALE_PER_TENSOR, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(valid_lhs_mode(rhs_mode), MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(E > 0 && E <= kMaxGroups && group_offset >= 0 && E_local > 0 && group_offset + E_local <= E,
                 MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(M >= 0 && M < (1ll << 31) && K > 0 && K % 16 == 0 && K < (1 << 30) && N > 0 && N % 16 == 0,
                 MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(static_cast<int64_t>(E_local) * N < (1ll << 31), MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(rhs_mode != MOE_SCALE_PER_ROW_BLOCK128 || K % 128 == 0, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(aligned16(lhs_q) && aligned16(rhs_q) && aligned16(out), MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(!workspace || (aligned16(workspace) && workspace_bytes >= gmm_fp8_w8_workspace_bytes(M, K)),
                 MOE_ERR_INVALID_ARG);
  // the 256-token tile when the local groups average 256 rows or more (the
  // full-rate N = 256 MMA), else the 128-token tile (less padding); with the
  // 256-token tile and a workspace the activations are decoded to f16 there
  // first (the 128-token tile serves small, weight-stream-bound groups, where
  // the extra pass costs more than it saves)
  const bool tok256 = M >= 256ll * E_local;
  const bool xf16 = workspace != nullptr && tok256;
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  if (M == 0) return MOE_OK;
  if (group_offset > 0 || E_local < E) {
    zero_outside_kernel<<<sm_count() * 4, 256, 0, st>>>(out, M, N, group_sizes, E, group_offset, E_local);
    MOE_CUDA_TRY(cudaGetLastError());
  }
  CUtensorMap X, W;
  if (xf16) {
    const int64_t n16 = M * K / 16;
    const int64_t blocks = std::min<int64_t>((n16 + 255) / 256, static_cast<int64_t>(sm_count()) * 8);
    e4m3_to_f16_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(lhs_q, n16, static_cast<uint16_t*>(workspace));
    MOE_CUDA_TRY(cudaGetLastError());
    // f16 rows of K elements, boxes of 128 rows x 64 elements (128-byte swizzle)
    if (!make_map_bf16(&X, workspace, K, M, 2 * K, 128)) return MOE_ERR_CUDA;
  } else if (!make_map_u8_64(&X, lhs_q, K, M, K, 128)) {
    return MOE_ERR_CUDA;
  }
  if (!make_map_u8_64(&W, rhs_q, K, static_cast<uint64_t>(E_local) * N, K, 128)) return MOE_ERR_CUDA;
  Params p{};
  p.group_sizes = group_sizes;
  p.E = E;
  p.g0 = group_offset;
  p.El = E_local;
  p.M = M;
  p.K = static_cast<int>(K);
  p.N = static_cast<int>(N);
  p.kblocks = static_cast<int>((K + BK - 1) / BK);
  p.lhs_scale = lhs_scale;
  p.lhs_mode = lhs_mode;
  p.rhs_scale = rhs_scale;
  p.rhs_mode = rhs_mode;
  p.out = out;
  p.stall_ns = g_stall_ns.load();
  p.stall = p.stall_ns != 0;
  if (tok256)
    return xf16 ? launch_w8<256, true>(X, W, p, E_local, st) : launch_w8<256, false>(X, W, p, E_local, st);
  return launch_w8<128, false>(X, W, p, E_local, st);
}

extern "C" size_t tgmm_fp8_workspace_bytes(int64_t M, int64_t K, int64_t N, int E_local) {
  if (M < 0 || K <= 0 || N <= 0 || E_local <= 0) return 0;
  const int64_t Mp = padded_rows(M, E_local);
  return align256(static_cast<size_t>(K * Mp)) + align256(static_cast<size_t>(N * Mp));
}

namespace moe {
namespace {
// tgmm_fp8 and tgmm_fp8_gcq: lay the rhs out (transposed and group-padded in
// the workspace) with `rhs_layout`, the lhs likewise from its codes, then
// contract over the padded rows.
template <class RhsLayout>
moe_status tgmm_run(const uint8_t* lhs_q, const float* lhs_scale, moe_scale_mode lhs_mode, const float* rhs_scale,
                    moe_scale_mode rhs_mode, const int32_t* group_sizes, int E, int group_offset, int E_local,
                    int64_t M, int64_t K, int64_t N, float* out, void* workspace, cudaStream_t st,
                    RhsLayout rhs_layout) {
  const int64_t Mp = padded_rows(M, E_local);
  uint8_t* lhsT = static_cast<uint8_t*>(workspace);
  uint8_t* rhsT = lhsT + align256(static_cast<size_t>(K * Mp));
  if (M > 0) {
    const int grid = sm_count() * 8;
    transpose_pad_kernel<<<grid, 256, 0, st>>>(lhs_q, M, K, lhsT, Mp, group_sizes, E, group_offset, E_local);
    MOE_CUDA_TRY(cudaGetLastError());
    rhs_layout(rhsT, Mp, grid);
    MOE_CUDA_TRY(cudaGetLastError());
  }
  CUtensorMap A, B;
  if (!make_map(&A, lhsT, Mp, K, Mp, BM)) return MOE_ERR_CUDA;
  constexpr int bn = Cfg<kTgmm>::BN;
  if (!make_map(&B, rhsT, Mp, N, Mp, bn)) return MOE_ERR_CUDA;
  Params p{};
  p.group_sizes = group_sizes;
  p.E = E;
  p.g0 = group_offset;
  p.El = E_local;
  p.M = M;
  p.K = static_cast<int>(K);
  p.N = static_cast<int>(N);
  p.kblocks = 0;
  p.ntiles = static_cast<int>((N + bn - 1) / bn);
  p.ktiles = static_cast<int>((K + BM - 1) / BM);
  p.lhs_scale = lhs_scale;
  p.lhs_mode = lhs_mode;
  p.rhs_scale = rhs_scale;
  p.rhs_mode = rhs_mode;
  p.out = out;
  const int64_t tiles = static_cast<int64_t>(E_local) * p.ktiles * p.ntiles;
  CUtensorMap O;
  if (!make_map_out_f32(&O, out, N, K, E_local)) return MOE_ERR_CUDA;
  return launch_mma<kTgmm, false>(A, B, O, p, static_cast<int>(tiles > (1 << 30) ? (1 << 30) : tiles), st);
}

#define MOE_TGMM_COMMON_CHECKS()                                                                               \
  MOE_HOST_CHECK((lhs_mode == MOE_SCALE_PER_TENSOR || lhs_mode == MOE_SCALE_PER_GROUP_COL), MOE_ERR_INVALID_ARG); \
  MOE_HOST_CHECK(E > 0 && E <= kMaxGroups && group_offset >= 0 && E_local > 0 && group_offset + E_local <= E,   \
                 MOE_ERR_INVALID_ARG);                                                                         \
  MOE_HOST_CHECK(M >= 0 && M < (1ll << 30) && K > 0 && K % 16 == 0 && K < (1 << 30) && N > 0 && N % 16 == 0 &&  \
                     N < (1 << 30),                                                                            \
                 MOE_ERR_INVALID_ARG);                                                                         \
  MOE_HOST_CHECK(aligned16(lhs_q) && aligned16(out) && aligned16(workspace), MOE_ERR_INVALID_ARG);             \
  MOE_HOST_CHECK(workspace_bytes >= tgmm_fp8_workspace_bytes(M, K, N, E_local), MOE_ERR_INVALID_ARG)
}  // namespace
}  // namespace moe

extern "C" moe_status tgmm_fp8(const uint8_t* lhs_q, const float* lhs_scale, moe_scale_mode lhs_mode,
                               const uint8_t* rhs_q, const float* rhs_scale, moe_scale_mode rhs_mode,
                               const int32_t* group_sizes, int E, int group_offset, int E_local, int64_t M,
                               int64_t K, int64_t N, float* out, void* workspace, size_t workspace_bytes,
                               moe_stream_t stream) {
  MOE_HOST_CHECK(lhs_q && lhs_scale && rhs_q && rhs_scale && group_sizes && out && workspace, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(rhs_mode == MOE_SCALE_PER_TENSOR || rhs_mode == MOE_SCALE_PER_GROUP_COL, MOE_ERR_INVALID_ARG);
  MOE_TGMM_COMMON_CHECKS();
  MOE_HOST_CHECK(aligned16(rhs_q) && (rhs_mode == MOE_SCALE_PER_TENSOR || aligned16(rhs_scale)), MOE_ERR_INVALID_ARG);
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  return tgmm_run(lhs_q, lhs_scale, lhs_mode, rhs_scale, rhs_mode, group_sizes, E, group_offset, E_local, M, K, N,
                  out, workspace, st, [&](uint8_t* rhsT, int64_t Mp, int grid) {
                    transpose_pad_kernel<<<grid, 256, 0, st>>>(rhs_q, M, N, rhsT, Mp, group_sizes, E, group_offset,
                                                               E_local);
                  });
}

extern "C" moe_status tgmm_fp8_gcq(const uint8_t* lhs_q, const float* lhs_scale, moe_scale_mode lhs_mode,
                                   const uint16_t* rhs_g, const float* rhs_scale, const int32_t* group_sizes, int E,
                                   int group_offset, int E_local, int64_t M, int64_t K, int64_t N, float* out,
                                   void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  MOE_HOST_CHECK(lhs_q && lhs_scale && rhs_g && rhs_scale && group_sizes && out && workspace, MOE_ERR_INVALID_ARG);
  MOE_TGMM_COMMON_CHECKS();
  MOE_HOST_CHECK(aligned16(rhs_g) && aligned16(rhs_scale), MOE_ERR_INVALID_ARG);
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  return tgmm_run(lhs_q, lhs_scale, lhs_mode, rhs_scale, MOE_SCALE_PER_GROUP_COL, group_sizes, E, group_offset,
                  E_local, M, K, N, out, workspace, st, [&](uint8_t* rhsT, int64_t Mp, int grid) {
                    quant_transpose_pad_kernel<<<grid, 256, 0, st>>>(rhs_g, M, N, rhs_scale, rhsT, Mp, group_sizes,
                                                                     E, group_offset, E_local);
                  });
}

// ---------------------------------------------------------------------------
// Router ("Support quantization for tokamax gmm v2", table 1: grad_gate-kernel
// and state_grad).  The gate contraction runs on the tcgen05 tensor cores in
// bf16 (kind::f16) with the softmax and top-k in its epilogue; the gradients'
// two contractions use the same kernel without scales.
// ---------------------------------------------------------------------------
extern "C" cudaError_t moe_detail_router_dw(const uint16_t* G, const uint16_t* o, const int32_t* pos, int64_t T,
                                            int k, int64_t D, float* dw, cudaStream_t st);
extern "C" cudaError_t moe_detail_router_dlogits(const float* logits, const int32_t* ids, const float* dw, int64_t T,
                                                 int E, int k, int Ep, int64_t Tp, uint16_t* dl, uint16_t* dl_pad,
                                                 uint16_t* dlT, cudaStream_t st);
extern "C" cudaError_t moe_detail_transpose_u16(const uint16_t* src, int64_t R, int64_t C, uint16_t* dst, int64_t Rp,
                                                cudaStream_t st);

namespace moe {
namespace {
constexpr int kRouterMaxE = 256;
constexpr int kRouterMaxK = 8;
int64_t round8(int64_t v) { return (v + 7) / 8 * 8; }

// out[M, N] = A[M, K] B[N, K]^T for bf16 row-major A and B (row pitches in
// elements), fp32 or bf16 out, on the tcgen05 kernel without scales.
moe_status bf16_gemm(const uint16_t* A, int64_t pitchA, const uint16_t* B, int64_t pitchB, int64_t M, int64_t N,
                     int64_t K, void* out, bool out_f32, cudaStream_t st) {
  if (M == 0 || N == 0) return MOE_OK;
  CUtensorMap ma, mb;
  if (!make_map_bf16(&ma, A, K, M, pitchA * 2, BM)) return MOE_ERR_CUDA;
  if (!make_map_bf16(&mb, B, K, N, pitchB * 2, Cfg<kBf16>::BN)) return MOE_ERR_CUDA;
  Params p{};
  p.group_sizes = nullptr;  // one group of M rows
  p.E = 1;
  p.g0 = 0;
  p.El = 1;
  p.M = M;
  p.K = static_cast<int>(K);
  p.N = static_cast<int>(N);
  p.kblocks = static_cast<int>((K + Cfg<kBf16>::KSTEP - 1) / Cfg<kBf16>::KSTEP);
  p.ntiles = static_cast<int>((N + Cfg<kBf16>::BN - 1) / Cfg<kBf16>::BN);
  p.out = out;
  p.out_f32 = out_f32 ? 1 : 0;
  return launch_mma<kBf16, false>(ma, mb, ma, p, gmm_max_units<kBf16, false>(M, 1, p.ntiles), st);
}
}  // namespace
}  // namespace moe

extern "C" moe_status moe_router_topk(const uint16_t* x, const uint16_t* w_gate, int64_t T, int64_t D, int E, int k,
                                      float* logits, int32_t* topk_ids, float* topk_w, moe_stream_t stream) {
  MOE_HOST_CHECK(x && w_gate && logits && topk_ids && topk_w, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(T >= 0 && T < (1ll << 31) && D > 0 && D % 8 == 0 && D < (1ll << 30), MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(E >= 1 && E <= kRouterMaxE && k >= 1 && k <= kRouterMaxK && k <= E, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(aligned16(x) && aligned16(w_gate), MOE_ERR_INVALID_ARG);
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  cudaStream_t st = as_stream(stream);
  CUtensorMap A, B;
  if (!make_map_bf16(&A, x, D, T, D * 2, BM)) return MOE_ERR_CUDA;
  // the gate's E rows, read as a 256-row box (rows past E come in as zeros)
  if (!make_map_bf16(&B, w_gate, D, E, D * 2, Cfg<kRouter>::BN)) return MOE_ERR_CUDA;
  Params p{};
  p.group_sizes = nullptr;
  p.E = 1;
  p.g0 = 0;
  p.El = 1;
  p.M = T;
  p.K = static_cast<int>(D);
  p.N = Cfg<kRouter>::BN;
  p.kblocks = static_cast<int>((D + Cfg<kRouter>::KSTEP - 1) / Cfg<kRouter>::KSTEP);
  p.ntiles = 1;
  p.rE = E;
  p.rk = k;
  p.logits = logits;
  p.topk_ids = topk_ids;
  p.topk_w = topk_w;
  return launch_mma<kRouter, false>(A, B, A, p, gmm_max_units<kRouter, false>(T, 1, 1), st);
}

namespace {
struct RouterWs {
  uint16_t *dl_pad, *dlT, *xT, *wgT;
};
size_t router_ws_layout(int64_t T, int64_t D, int E, RouterWs* w, void* base) {
  const int64_t Tp = moe::round8(T), Ep = moe::round8(E);
  const size_t sizes[4] = {static_cast<size_t>(T * Ep) * 2, static_cast<size_t>(Ep * Tp) * 2,
                           static_cast<size_t>(D * Tp) * 2, static_cast<size_t>(D * Ep) * 2};
  size_t off = 0;
  uint16_t* ptrs[4];
  for (int i = 0; i < 4; ++i) {
    ptrs[i] = base ? reinterpret_cast<uint16_t*>(static_cast<char*>(base) + off) : nullptr;
    off += (sizes[i] + 255) & ~static_cast<size_t>(255);
  }
  if (w) *w = RouterWs{ptrs[0], ptrs[1], ptrs[2], ptrs[3]};
  return off;
}
}  // namespace

extern "C" size_t moe_router_backward_workspace_bytes(int64_t T, int64_t D, int E) {
  if (T < 0 || D <= 0 || E <= 0) return 0;
  return router_ws_layout(T, D, E, nullptr, nullptr);
}

extern "C" moe_status moe_router_backward(const uint16_t* G, const uint16_t* o, const int32_t* pos, const uint16_t* x,
                                          const uint16_t* w_gate, const float* logits, const int32_t* topk_ids,
                                          int64_t T, int64_t D, int E, int k, float* dw, uint16_t* dlogits,
                                          float* grad_gate, uint16_t* state_grad, void* workspace,
                                          size_t workspace_bytes, moe_stream_t stream) {
  MOE_HOST_CHECK(G && o && pos && x && w_gate && logits && topk_ids && dw && dlogits && grad_gate && state_grad &&
                     workspace,
                 MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(T >= 0 && T <= (1ll << 21) && D > 0 && D % 16 == 0 && D < (1ll << 30), MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(E >= 1 && E <= kRouterMaxE && k >= 1 && k <= kRouterMaxK && k <= E, MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(aligned16(G) && aligned16(o) && aligned16(x) && aligned16(w_gate) && aligned16(grad_gate) &&
                     aligned16(state_grad) && aligned16(workspace),
                 MOE_ERR_INVALID_ARG);
  MOE_HOST_CHECK(workspace_bytes >= moe_router_backward_workspace_bytes(T, D, E), MOE_ERR_INVALID_ARG);
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  if (T == 0) {
    MOE_CUDA_TRY(cudaMemsetAsync(grad_gate, 0, sizeof(float) * static_cast<size_t>(E) * D, st));
    return MOE_OK;
  }
  RouterWs w;
  router_ws_layout(T, D, E, &w, workspace);
  const int64_t Tp = round8(T), Ep = round8(E);
  MOE_CUDA_TRY(moe_detail_router_dw(G, o, pos, T, k, D, dw, st));
  MOE_CUDA_TRY(moe_detail_router_dlogits(logits, topk_ids, dw, T, E, k, static_cast<int>(Ep), Tp, dlogits, w.dl_pad,
                                         w.dlT, st));
  MOE_CUDA_TRY(moe_detail_transpose_u16(x, T, D, w.xT, Tp, st));
  MOE_CUDA_TRY(moe_detail_transpose_u16(w_gate, E, D, w.wgT, Ep, st));
  // grad_gate [E, D] = dlogits^T x: rows of dlT against rows of xT, K = T
  moe_status stt = bf16_gemm(w.dlT, Tp, w.xT, Tp, E, D, T, grad_gate, true, st);
  if (stt != MOE_OK) return stt;
  // state_grad [T, D] = dlogits W_gate: rows of dlogits against rows of W_gate^T, K = E
  return bf16_gemm(w.dl_pad, Ep, w.wgT, Ep, T, D, E, state_grad, false, st);
}
