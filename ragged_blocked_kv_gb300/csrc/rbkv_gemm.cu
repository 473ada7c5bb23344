// The dense steps of a decoder layer around the attention pass: a bf16 GEMM
// on the fifth-generation tensor cores with fused epilogues, and RMSNorm.
//
// DeepSpeed-FastGen paper summary page, idea I1: the latency of a forward pass
// follows the number of tokens in it; the token-proportional work of a layer
// is its projections (QKV, output, and the two MLP products), matrix products
// of the pass's [T][hidden] activations with the layer's weights.
//
// GEMM: C[M][N] = A[M][K] . B[N][K]^T (both operands K-major: activations are
// rows of K values, weights are stored [out][in]), bf16 in, fp32 accumulation
// in tensor memory, bf16 out.  Epilogues: plain; + R (a residual [M][N]);
// SwiGLU, where B's rows come in blocks of 256 - 128 gate rows, then the 128
// up rows of the same outputs - and C[M][N/2] = silu(gate) * up; or a split of
// C's columns into three row-major outputs (Q, K and V of a QKV projection).
// Design: tiles of 128 x 256 outputs (one tcgen05.mma M=128 N=256 K=16 per
// 16 of K), K in steps of 64 (one 128-byte swizzle row of bf16) through a
// 4-stage TMA ring of 48 KB; a persistent grid of one CTA per SM walks the
// tiles (the M tiles of one N tile next to each other, so a weight tile is
// read from HBM once and from L2 by the others); two accumulators in tensor
// memory (2 x 256 columns) so that a tile's epilogue overlaps the next tile's
// products.  Warp 0 loads, warp 1 issues the MMAs, warps 2-5 (one TMEM lane
// quadrant each) run the epilogue.  Every wait is bounded.
// Schedule: whole waves of tiles run as whole tiles; when the tiles that are
// left would fill a last wave only in part, their K range is split into
// pieces spread over all SMs (fp32 partials in a caller workspace, summed and
// finished by a second kernel).  With fewer tiles than SMs, every tile is
// split.  The tiles left over are the last column blocks (tiles are numbered
// with the M tiles of one weight tile next to each other), so the partials
// cover only those columns.
#include <algorithm>
#include <atomic>

#include "rbkv_internal.h"
#include "rbkv_ptx.cuh"
#include "rbkv_tcgen05.cuh"

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace rbkv {

namespace {

using namespace tc;

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;            // 16 KB
constexpr int kBBytes = kBN * kBK * 2;            // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;    // 48 KB
constexpr int kThreads = 6 * 32;
constexpr int kAccCols = kBN;                     // fp32 columns of one accumulator
constexpr int kSmemBytes = kStages * kStageBytes + 1024;
constexpr long long kWaitLimit = 4000000000LL;

struct GemmBars {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(kStages * kStageBytes + (int)sizeof(GemmBars) <= kSmemBytes, "smem layout");

struct GemmArgs {
  __nv_bfloat16* c;
  __nv_bfloat16* c2;          // split epilogue: the second and third outputs
  __nv_bfloat16* c3;
  int32_t split1, split2;     // split epilogue: first columns of the second and third
  const __nv_bfloat16* r;     // residual (epilogue 1)
  int32_t* status;            // error word (wait timeouts), may be null
  int32_t M, N, K;
  int32_t ldc;                // row stride of C (and R) in elements
  int32_t epilogue;           // 0 plain, 1 residual, 2 SwiGLU, 3 split into three outputs
  int32_t m_tiles, n_tiles;
  int32_t full;               // tiles 0 .. full-1 run whole (a multiple of m_tiles)
  int32_t splits;             // the other tiles' K in this many pieces (1: none left)
  int32_t kps;                // k steps per piece
  int32_t tail_col0;          // first column of the split tiles: (full / m_tiles) * kBN
  float* ws;                  // fp32 partials [splits][M][N - tail_col0]
};

// Work unit u: a whole tile (u < full) or one K piece of a split tile.
struct Unit {
  int tile, piece, k_begin, k_end;
  bool partial;
};
__device__ __forceinline__ Unit unit_of(const GemmArgs& g, int u, int k_steps) {
  Unit x;
  if (u < g.full) {
    x.tile = u;
    x.piece = 0;
    x.k_begin = 0;
    x.k_end = k_steps;
    x.partial = false;
  } else {
    const int v = u - g.full;
    x.tile = g.full + v / g.splits;
    x.piece = v % g.splits;
    x.k_begin = x.piece * g.kps;
    x.k_end = min(k_steps, x.k_begin + g.kps);
    x.partial = true;
  }
  return x;
}

__device__ __forceinline__ float silu(float g) { return g / (1.f + __expf(-g)); }

__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_tcgen05_kernel(const __grid_constant__ CUtensorMap tmap_a,
                             const __grid_constant__ CUtensorMap tmap_b, GemmArgs g) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (ptx::smem_u32(smem_raw) & 1023) {
    if (threadIdx.x == 0 && g.status) atomicCAS(g.status, 0, kDevBounds);
    return;
  }
  GemmBars* bars = reinterpret_cast<GemmBars*>(smem_raw + kStages * kStageBytes);
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int units = g.full + (g.m_tiles * g.n_tiles - g.full) * g.splits;
  const int k_steps = (g.K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&bars->full[s], 1);
      ptx::mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&bars->acc_full[b], 1);
      ptx::mbar_init(&bars->acc_empty[b], 4 * 32);
    }
    bars->abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 2 * kAccCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // tile t: M tile t % m_tiles, N tile t / m_tiles (the M tiles of one weight
  // tile next to each other); CTA c takes tiles c, c + grid, ...

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmap_a);
      ptx::tma_prefetch_desc(&tmap_b);
      uint32_t it = 0;
      bool stop = false;
      for (int u = blockIdx.x; u < units && !stop; u += gridDim.x) {
        const Unit w = unit_of(g, u, k_steps);
        const int m0 = (w.tile % g.m_tiles) * kBM, n0 = (w.tile / g.m_tiles) * kBN;
        for (int ks = w.k_begin; ks < w.k_end; ++ks, ++it) {
          const int s = it % kStages;
          if (*abort_flag) {
            stop = true;
            break;
          }
          if (it >= (uint32_t)kStages &&
              !ptx::mbar_wait(&bars->empty[s], ((it / kStages) - 1) & 1, kWaitLimit)) {
            if (g.status) ptx::report_wait(g.status, kDevTimeout, 61, (int)it);
            *abort_flag = 1;
            stop = true;
            break;
          }
          uint8_t* a_dst = smem_raw + s * kStageBytes;
          uint8_t* b_dst = a_dst + kABytes;
          ptx::mbar_arrive_expect_tx(&bars->full[s], kStageBytes);
          ptx::tma_load_2d(a_dst, &tmap_a, ks * kBK, m0, &bars->full[s]);
          ptx::tma_load_2d(b_dst, &tmap_b, ks * kBK, n0, &bars->full[s]);
        }
      }
      for (uint32_t t = it > (uint32_t)kStages ? it - kStages : 0; t < it; ++t)
        ptx::mbar_wait(&bars->full[t % kStages], (t / kStages) & 1, kWaitLimit);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = instr_desc(kBM, kBN, 0);
      const uint32_t base_lo = desc_lo(ptx::smem_u32(smem_raw), 16);
      const uint32_t hi = desc_hi(1024);
      uint32_t it = 0, n = 0;
      bool ok = true;
      int site = 0, at = 0;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++n) {
        const Unit w = unit_of(g, u, k_steps);
        const int k_begin = w.k_begin, k_end = w.k_end;
        const uint32_t buf = n & 1;
        // the epilogue must have read this accumulator's previous tile
        if (n >= 2 && (!ptx::mbar_wait(&bars->acc_empty[buf], ((n >> 1) - 1) & 1, kWaitLimit) ||
                       *abort_flag)) {
          ok = false;
          site = 62;
          at = (int)n;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + buf * kAccCols;
        for (int ks = k_begin; ks < k_end; ++ks, ++it) {
          const int s = it % kStages;
          if (!ptx::mbar_wait(&bars->full[s], (it / kStages) & 1, kWaitLimit) || *abort_flag) {
            ok = false;
            site = 63;
            at = (int)it;
            break;
          }
          tc_fence_after();
          // descriptor low words of this stage's A and B tiles (the high word
          // is common); each 16-column step adds 32 bytes (2 in address units)
          const uint32_t a_lo = base_lo + ((s * kStageBytes) >> 4);
          const uint32_t b_lo = a_lo + (kABytes >> 4);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            tc_mma_ss_w(d, a_lo + kk * 2, b_lo + kk * 2, hi, idesc, ks > k_begin || kk > 0);
          tc_commit(&bars->empty[s]);
        }
        if (!ok) break;
        tc_commit(&bars->acc_full[buf]);
      }
      if (!ok) {
        if (g.status) ptx::report_wait(g.status, kDevTimeout, site, at);
        *abort_flag = 1;
      }
      // every MMA must finish before tensor memory is released
      if (n > 0) {
        const uint32_t last = n - 1;
        ptx::mbar_wait(&bars->acc_full[last & 1], (last >> 1) & 1, kWaitLimit);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;                         // TMEM lane quadrant of this warp
    const int row_in_tile = quad * 32 + lane;
    uint32_t n = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++n) {
      const Unit w = unit_of(g, u, k_steps);
      const int t = w.tile, piece = w.piece;
      const uint32_t buf = n & 1;
      const bool got = ptx::mbar_wait(&bars->acc_full[buf], (n >> 1) & 1, kWaitLimit);
      if (!__all_sync(0xffffffffu, got) || __any_sync(0xffffffffu, *abort_flag != 0)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int m0 = (t % g.m_tiles) * kBM, n0 = (t / g.m_tiles) * kBN;
      const int row = m0 + row_in_tile;
      const bool live = row < g.M;
      const uint32_t taddr = tmem + buf * kAccCols + ((uint32_t)(quad * 32) << 16);
      if (w.partial) {
        // one piece of K: the fp32 partial sums go to the workspace; the
        // reduce kernel adds the pieces and applies the epilogue
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          float v[32];
          tmem_ld32(taddr + c * 32, v);
          tmem_wait_ld();
          const int col = n0 + c * 32;
          if (live && col < g.N) {
            const int tail_cols = g.N - g.tail_col0;
            float4* dst = reinterpret_cast<float4*>(
                g.ws + ((int64_t)piece * g.M + row) * tail_cols + (col - g.tail_col0));
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          }
        }
      } else if (g.epilogue == 2) {
        // SwiGLU: columns 0..127 of the tile are gates, 128..255 the ups of
        // the same outputs n0 / 2 + 0..127
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float gv[32], uv[32];
          tmem_ld32(taddr + c * 32, gv);
          tmem_ld32(taddr + 128 + c * 32, uv);
          tmem_wait_ld();
          const int col = n0 / 2 + c * 32;
          if (live && col < g.N / 2) {
            __nv_bfloat16* dst = g.c + (int64_t)row * g.ldc + col;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 w;
              w.x = ptx::pack_bf16x2(silu(gv[v * 8 + 0]) * uv[v * 8 + 0], silu(gv[v * 8 + 1]) * uv[v * 8 + 1]);
              w.y = ptx::pack_bf16x2(silu(gv[v * 8 + 2]) * uv[v * 8 + 2], silu(gv[v * 8 + 3]) * uv[v * 8 + 3]);
              w.z = ptx::pack_bf16x2(silu(gv[v * 8 + 4]) * uv[v * 8 + 4], silu(gv[v * 8 + 5]) * uv[v * 8 + 5]);
              w.w = ptx::pack_bf16x2(silu(gv[v * 8 + 6]) * uv[v * 8 + 6], silu(gv[v * 8 + 7]) * uv[v * 8 + 7]);
              reinterpret_cast<uint4*>(dst)[v] = w;
            }
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          float v[32];
          tmem_ld32(taddr + c * 32, v);
          tmem_wait_ld();
          const int col = n0 + c * 32;
          if (live && col < g.N) {
            __nv_bfloat16* dst;
            if (g.epilogue == 3) {
              // columns [0, split1) to c, [split1, split2) to c2, the rest to c3,
              // each its own row-major matrix
              dst = col < g.split1 ? g.c + (int64_t)row * g.split1 + col
                    : col < g.split2 ? g.c2 + (int64_t)row * (g.split2 - g.split1) + (col - g.split1)
                                     : g.c3 + (int64_t)row * (g.N - g.split2) + (col - g.split2);
            } else {
              dst = g.c + (int64_t)row * g.ldc + col;
            }
            if (g.epilogue == 1) {
              const uint4* rs = reinterpret_cast<const uint4*>(g.r + (int64_t)row * g.ldc + col);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const uint4 rv = rs[q];
                const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  v[q * 8 + 2 * e] += __uint_as_float(rw[e] << 16);
                  v[q * 8 + 2 * e + 1] += __uint_as_float(rw[e] & 0xffff0000u);
                }
              }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 w;
              w.x = ptx::pack_bf16x2(v[q * 8 + 0], v[q * 8 + 1]);
              w.y = ptx::pack_bf16x2(v[q * 8 + 2], v[q * 8 + 3]);
              w.z = ptx::pack_bf16x2(v[q * 8 + 4], v[q * 8 + 5]);
              w.w = ptx::pack_bf16x2(v[q * 8 + 6], v[q * 8 + 7]);
              reinterpret_cast<uint4*>(dst)[q] = w;
            }
          }
        }
      }
      tc_fence_before();
      ptx::mbar_arrive(&bars->acc_empty[buf]);
    }
    if (!ok && lane == 0 && g.status) ptx::report_wait(g.status, kDevTimeout, 64, (int)n);
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kAccCols);
  }
}

// ---------------------------------------------------------------------------
// Split-K reduction: the pieces' fp32 partials summed, then the epilogue
// ---------------------------------------------------------------------------
// Thread i takes 8 consecutive outputs of C in the split tiles' columns (of
// the SwiGLU output for epilogue 2: the 8 gates and the 8 ups of those
// outputs).
__global__ void __launch_bounds__(256) gemm_splitk_reduce_kernel(GemmArgs g) {
  const int out_n = g.epilogue == 2 ? g.N / 2 : g.N;
  const int out_c0 = g.epilogue == 2 ? g.tail_col0 / 2 : g.tail_col0;
  const int tail_cols = g.N - g.tail_col0;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t per_row = (out_n - out_c0) / 8;
  if (i >= (int64_t)g.M * per_row) return;
  const int row = (int)(i / per_row), j0 = out_c0 + (int)(i % per_row) * 8;
  const int64_t piece_stride = (int64_t)g.M * tail_cols;
  auto sum8 = [&](int col, float* v) {
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = 0.f;
    const float* src = g.ws + (int64_t)row * tail_cols + (col - g.tail_col0);
    for (int p = 0; p < g.splits; ++p) {
      const float4 a = *reinterpret_cast<const float4*>(src + p * piece_stride);
      const float4 b = *reinterpret_cast<const float4*>(src + p * piece_stride + 4);
      v[0] += a.x; v[1] += a.y; v[2] += a.z; v[3] += a.w;
      v[4] += b.x; v[5] += b.y; v[6] += b.z; v[7] += b.w;
    }
  };
  float v[8];
  __nv_bfloat16* dst;
  if (g.epilogue == 2) {
    const int blk = j0 / 128, jj = j0 % 128;
    float u[8];
    sum8(blk * 256 + jj, v);
    sum8(blk * 256 + 128 + jj, u);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = silu(v[e]) * u[e];
    dst = g.c + (int64_t)row * g.ldc + j0;
  } else {
    sum8(j0, v);
    if (g.epilogue == 1) {
      const uint4 rv = *reinterpret_cast<const uint4*>(g.r + (int64_t)row * g.ldc + j0);
      const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[2 * e] += __uint_as_float(rw[e] << 16);
        v[2 * e + 1] += __uint_as_float(rw[e] & 0xffff0000u);
      }
    }
    if (g.epilogue == 3) {
      const int col = j0;
      dst = col < g.split1 ? g.c + (int64_t)row * g.split1 + col
            : col < g.split2 ? g.c2 + (int64_t)row * (g.split2 - g.split1) + (col - g.split1)
                             : g.c3 + (int64_t)row * (g.N - g.split2) + (col - g.split2);
    } else {
      dst = g.c + (int64_t)row * g.ldc + j0;
    }
  }
  uint4 w;
  w.x = ptx::pack_bf16x2(v[0], v[1]);
  w.y = ptx::pack_bf16x2(v[2], v[3]);
  w.z = ptx::pack_bf16x2(v[4], v[5]);
  w.w = ptx::pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(dst) = w;
}

// ---------------------------------------------------------------------------
// RMSNorm: y[m][:] = x[m][:] / sqrt(mean(x[m][:]^2) + eps) * w[:], one warp a row
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
    rmsnorm_bf16_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ w,
                        __nv_bfloat16* __restrict__ y, int32_t M, int32_t H, float eps) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= M) return;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (int64_t)warp * H);
  const int vec = H / 8;
  float ss = 0.f;
  for (int i = lane; i < vec; i += 32) {
    const uint4 u = xr[i];
    const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a = __uint_as_float(uw[e] << 16), b = __uint_as_float(uw[e] & 0xffff0000u);
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
    }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float inv = rsqrtf(ss / (float)H + eps);
  const uint4* wr = reinterpret_cast<const uint4*>(w);
  uint4* yr = reinterpret_cast<uint4*>(y + (int64_t)warp * H);
  for (int i = lane; i < vec; i += 32) {
    const uint4 u = xr[i], gw = wr[i];
    const uint32_t uw[4] = {u.x, u.y, u.z, u.w}, ww[4] = {gw.x, gw.y, gw.z, gw.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a = __uint_as_float(uw[e] << 16) * inv * __uint_as_float(ww[e] << 16);
      const float b = __uint_as_float(uw[e] & 0xffff0000u) * inv *
                      __uint_as_float(ww[e] & 0xffff0000u);
      o[e] = ptx::pack_bf16x2(a, b);
    }
    yr[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

int sms_of_current(cudaError_t* err) {
  static int sms_of[64] = {0};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return 0;
  int sms = dev < 64 ? sms_of[dev] : 0;
  if (sms == 0) {
    *err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (*err != cudaSuccess) return 0;
    if (dev < 64) sms_of[dev] = sms;
  }
  return sms;
}

}  // namespace

// How a product is scheduled over `sms` SMs: the tiles that run whole, the
// pieces each other tile's K is split into, and the k steps of a piece.
struct GemmPlan {
  int64_t full, splits, kps, tail_col0;
};

GemmPlan gemm_plan(int64_t M, int64_t N, int64_t K, int sms) {
  const int64_t m_tiles = (M + kBM - 1) / kBM, n_tiles = (N + kBN - 1) / kBN;
  const int64_t tiles = m_tiles * n_tiles, k_steps = (K + kBK - 1) / kBK;
  const GemmPlan whole{tiles, 1, k_steps, N};
  if (sms <= 0) return whole;
  // the tiles of whole waves run whole (rounded down to whole column blocks);
  // the rest are split into enough pieces to give every SM a unit, each at
  // least 8 k steps long
  const int64_t full = tiles < sms ? 0 : (tiles / sms) * sms / m_tiles * m_tiles;
  const int64_t tail = tiles - full;
  if (tail == 0) return whole;
  int64_t s = std::min<int64_t>({(int64_t)sms / tail, k_steps / 8, 16});
  if (s < 2) return whole;
  const int64_t kps = (k_steps + s - 1) / s;
  s = (k_steps + kps - 1) / kps;   // no empty piece
  // k steps on the busiest SM, whole tiles against the split schedule (the
  // grid walks units b, b + G, ...; the reduce kernel's pass comes on top)
  auto busiest = [&](int64_t f, int64_t pieces, int64_t per_piece) {
    const int64_t units = f + (tiles - f) * pieces;
    const int64_t G = std::min<int64_t>(units, sms);
    int64_t worst = 0;
    for (int64_t b = 0; b < G; ++b) {
      int64_t load = 0;
      for (int64_t u = b; u < units; u += G) load += u < f ? k_steps : per_piece;
      worst = std::max(worst, load);
    }
    return worst;
  };
  if (10 * busiest(full, s, kps) > 9 * busiest(tiles, 1, k_steps)) return whole;
  return GemmPlan{full, s, kps, full / m_tiles * kBN};
}

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  cudaError_t e;
  const int sms = sms_of_current(&e);
  if (e != cudaSuccess || sms <= 0) return 0;
  const GemmPlan p = gemm_plan(M, N, K, sms);
  return p.splits > 1 ? (size_t)p.splits * M * (N - p.tail_col0) * sizeof(float) : 0;
}

cudaError_t launch_gemm_bf16(const void* a, const void* b, void* c, const void* r, int64_t M,
                             int64_t N, int64_t K, int64_t ldc, int epilogue, int32_t* status,
                             cudaStream_t st, void* c2, void* c3, int64_t split1, int64_t split2,
                             void* ws, size_t ws_bytes) {
  if (M <= 0 || N <= 0 || K <= 0) return cudaSuccess;
  CUtensorMap ta, tb;
  cudaError_t e = make_tmap_2d(&ta, a, M, K, kBM);
  if (e == cudaSuccess) e = make_tmap_2d(&tb, b, N, K, kBN);
  if (e != cudaSuccess) return e;
  static std::atomic<uint64_t> attr_done{0};
  const int sms = sms_of_current(&e);
  if (e != cudaSuccess) return e;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done.load() & bit)) {
    e = cudaFuncSetAttribute(gemm_bf16_tcgen05_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit);
  }
  GemmArgs g;
  g.c = (__nv_bfloat16*)c;
  g.c2 = (__nv_bfloat16*)c2;
  g.c3 = (__nv_bfloat16*)c3;
  g.split1 = (int32_t)split1;
  g.split2 = (int32_t)split2;
  g.r = (const __nv_bfloat16*)r;
  g.status = status;
  g.M = (int32_t)M;
  g.N = (int32_t)N;
  g.K = (int32_t)K;
  g.ldc = (int32_t)ldc;
  g.epilogue = epilogue;
  g.m_tiles = (int32_t)((M + kBM - 1) / kBM);
  g.n_tiles = (int32_t)((N + kBN - 1) / kBN);
  const int64_t k_steps = (K + kBK - 1) / kBK;
  // the split schedule needs the caller's workspace; without one (or with
  // one too small) every tile runs whole
  GemmPlan plan = gemm_plan(M, N, K, sms);
  if (!ws || (plan.splits > 1 && ws_bytes < (size_t)plan.splits * M * (N - plan.tail_col0) *
                                                sizeof(float)))
    plan = GemmPlan{(int64_t)g.m_tiles * g.n_tiles, 1, k_steps, N};
  g.full = (int32_t)plan.full;
  g.splits = (int32_t)plan.splits;
  g.kps = (int32_t)plan.kps;
  g.tail_col0 = (int32_t)plan.tail_col0;
  g.ws = (float*)ws;
  const int64_t units = plan.full + ((int64_t)g.m_tiles * g.n_tiles - plan.full) * plan.splits;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min<int64_t>(units, std::max(1, sms)));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  e = cudaLaunchKernelEx(&cfg, gemm_bf16_tcgen05_kernel, ta, tb, g);
  if (e != cudaSuccess || g.splits == 1) return e;
  const int64_t threads = M * ((epilogue == 2 ? (N - plan.tail_col0) / 2 : N - plan.tail_col0) / 8);
  gemm_splitk_reduce_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(g);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_bf16(const void* x, const void* w, void* y, int64_t M, int64_t H,
                                float eps, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  const int64_t threads = M * 32;
  rmsnorm_bf16_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(
      (const __nv_bfloat16*)x, (const __nv_bfloat16*)w, (__nv_bfloat16*)y, (int32_t)M,
      (int32_t)H, eps);
  return cudaGetLastError();
}

}  // namespace rbkv
