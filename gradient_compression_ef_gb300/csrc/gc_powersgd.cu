// gc_powersgd.cu -- one rank-r PowerSGD step with error feedback.
//
// "gradient-compression-quantization-sparsification" 3.1 (low-rank
// approximation: send two thin matrices, rebuild on the receiver) and
// Vogels et al., NeurIPS 2019, Algorithm 1:
//   M = G + E;  P = M Q;  P_hat = orthonormalise(P);  Q' = M^T P_hat;
//   E' = M - P_hat Q'^T.
//
// At rank r the step moves >= 12 bytes per element and performs 6r flops
// per element: about 2 flop/byte at r = 4, two orders of magnitude below
// the tensor-core ridge point, so every pass is organised around HBM
// streaming.  Two paths:
//
// Rows of a 16-byte multiple (n % 4 == 0): pass 1 (M = G + E, P = M Q)
// runs on the tensor cores (tcgen05, TF32 in three products), passes 2 and
// 3 on the CUDA cores; W = U^-1 and P_hat = P W are formed inside pass 2
// and the final reduction of Q' is a small grid of its own.  The section
// "Tensor-core path" below describes it.
//
// Other column counts, all on the CUDA cores:
//   pass 1  mq       : M = G + E written over E; P = M Q (Q staged in shared
//                      memory).  Blocks own 16 rows and a range of columns
//                      (enough blocks to fill the GPU); the last block of a
//                      row range adds the column ranges' partial rows of P in
//                      order and forms their Gram matrix in fp64.  The last
//                      row range sums the Gram partials in order, factors
//                      P^T P = U^T U (Cholesky, fp64, one warp) and stores
//                      W = U^-1.  P W is the Gram-Schmidt orthonormalisation
//                      of P: both give the unique QR factor with a positive
//                      diagonal.
//   pass 2  mtp      : Q' = M^T P_hat.  Blocks own a 128-column strip and a
//                      slice of rows; P_hat = P W for the slice is formed in
//                      shared memory (strip 0 also writes it out).  Partial
//                      sums are reduced in a fixed order by the last block of
//                      each strip, so results are deterministic.
//   pass 3  residual : E' = M - P_hat Q'^T (Q' staged in shared memory),
//                      blocks over rows and column ranges as in pass 1.
// Traffic: 12 + 4 + 8 = 24 bytes per element.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "gc_internal.cuh"
#include "gc_sm100.cuh"

namespace gc {
namespace {

constexpr int kPThreads = 256;
constexpr int kPWarps = kPThreads / 32;
constexpr int kRowsPerWarp = 2;
constexpr int kRowsPerBlock = kPWarps * kRowsPerWarp;  // 16
constexpr int kQChunk = 512;                           // columns of Q per stage
constexpr int kStrip = 128;                            // columns per pass-2 block
constexpr int kPhRows = 512;                           // P_hat rows staged per pass-2 step
constexpr int kMaxColSplits = 8;                       // column ranges of passes 1 and 3
constexpr int kSubSteps = 2;                           // 128-column steps loaded together

struct PsgdState {
  uint32_t ticket_mq;
  uint32_t pad[3];
};

struct PsgdBufs {
  float* praw;        // [m][r] raw P
  float* ppart;       // [splits][m][r] partial rows of P per column range
  uint32_t* rb_tickets;  // [row blocks] last-block tickets of pass 1
  double* gram_part;  // [blocks][r][r]
  float* w;           // [r][r] W = U^-1 (upper triangular)
  float* q_part;      // [splits][n][r]
  uint32_t* tickets;  // [strips]
  PsgdState* state;
  uint32_t* status;
};

template <bool VEC>
__device__ __forceinline__ void load_row4(const float* row, int64_t j, int64_t n, float v[4]) {
  if (VEC && j + 3 < n) {
    const float4 t = *reinterpret_cast<const float4*>(row + j);
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = (j + q < n) ? row[j + q] : 0.0f;
  }
}

template <bool VEC>
__device__ __forceinline__ void store_row4(float* row, int64_t j, int64_t n, const float v[4]) {
  if (VEC && j + 3 < n) {
    *reinterpret_cast<float4*>(row + j) = make_float4(v[0], v[1], v[2], v[3]);
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (j + q < n) row[j + q] = v[q];
  }
}

// Stages Q[col0 .. col0 + kQChunk) (rows of the n x R matrix) in smem.
template <int R>
__device__ __forceinline__ void stage_q(float* qs, const float* Q, int64_t col0, int64_t n) {
  const int64_t cols = std::min<int64_t>(kQChunk, n - col0);
  const float* src = Q + col0 * R;
  for (int64_t t = threadIdx.x; t < (int64_t)kQChunk * R; t += kPThreads)
    qs[t] = t < cols * R ? src[t] : 0.0f;
}

// Cholesky P^T P = U^T U (U upper, positive diagonal) of the binary64 Gram
// matrix, and w = U^-1 (upper triangular, row-major R x R floats): P U^-1 is
// the orthonormal factor Gram-Schmidt gives.  A column whose remaining norm
// is 0 is dropped (its P_hat column is left zero), as Gram-Schmidt leaves a
// zero column zero.
//
// One warp, in shared memory: A (R x R, the Gram matrix, overwritten by U
// in its upper triangle) and rinv (R doubles).  Step k takes the pivot d =
// A[k][k], scales row k by 1 / sqrt(d) and subtracts the outer product of
// the scaled row from the trailing block, so every entry loses the same
// products in the same order as in the column-by-column form; the one
// reciprocal square root per pivot replaces the square root and the
// divisions (binary64 division and square root are long instruction
// sequences here, and the chain is serial).  Then lane j forms column j of
// W by back substitution.
template <int R>
__device__ void cholesky_inverse_warp(double* A, double* rinv, float* w, int lane) {
#pragma unroll 1
  for (int k = 0; k < R; ++k) {
    const double d = A[k * R + k];
    const bool z = !(d > 0.0);
    const double r = z ? 0.0 : rsqrt(d);
    __syncwarp();
    for (int j = k + 1 + lane; j < R; j += 32) A[k * R + j] = z ? 0.0 : A[k * R + j] * r;
    if (lane == 0) rinv[k] = r;  // 0 marks a dropped direction
    __syncwarp();
    const int T = R - 1 - k;
    for (int t = lane; t < T * T; t += 32) {
      const int i = k + 1 + t / T, j = k + 1 + t % T;
      if (i <= j) A[i * R + j] = A[i * R + j] - A[k * R + i] * A[k * R + j];
    }
    __syncwarp();
  }
  if (lane < R) {
    const int j = lane;
    double wc[R];
#pragma unroll
    for (int i = 0; i < R; ++i) wc[i] = 0.0;
    const double rj = rinv[j];
    if (rj != 0.0) {
#pragma unroll
      for (int i = R - 1; i >= 0; --i) {
        if (i == j) wc[i] = rj;
        const double ri = rinv[i];
        if (i < j && ri != 0.0) {
          double sum = 0.0;
#pragma unroll
          for (int k = 0; k < R; ++k)
            if (k > i && k <= j) sum += A[i * R + k] * wc[k];
          wc[i] = -sum * ri;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < R; ++i) w[i * R + j] = (float)wc[i];
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// pass 1: M = G + E, P = M Q, Gram partials; last block: W = chol(P^T P)^-1.
// ---------------------------------------------------------------------------
template <int R, bool VEC>
__global__ void __launch_bounds__(kPThreads) psgd_mq_kernel(
    const float* __restrict__ G, float* __restrict__ E, int64_t m, int64_t n,
    const float* __restrict__ Q, PsgdBufs b, int64_t cols_per_split) {
  __shared__ float qs[kQChunk * R];
  __shared__ float prow[kRowsPerBlock][R];
  __shared__ double gram[R * R];
  __shared__ double rinv[R];
  __shared__ bool last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t row0 = (int64_t)blockIdx.x * kRowsPerBlock + warp * kRowsPerWarp;
  const int split = blockIdx.y, splits = gridDim.y;
  const int64_t c_lo = (int64_t)split * cols_per_split;
  const int64_t c_hi = std::min<int64_t>(n, c_lo + cols_per_split);
  float acc[kRowsPerWarp][R];
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr)
#pragma unroll
    for (int c = 0; c < R; ++c) acc[rr][c] = 0.0f;

  for (int64_t col0 = c_lo; col0 < c_hi; col0 += kQChunk) {
    __syncthreads();
    stage_q<R>(qs, Q, col0, n);
    __syncthreads();
    // two 128-column steps of both rows loaded before any store (the
    // stores to E would otherwise order the next loads behind them)
#pragma unroll
    for (int s = 0; s < kQChunk / 128; s += kSubSteps) {
      float g[kSubSteps][kRowsPerWarp][4], e[kSubSteps][kRowsPerWarp][4];
#pragma unroll
      for (int u = 0; u < kSubSteps; ++u) {
        const int64_t j = col0 + (s + u) * 128 + 4 * lane;
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
          const int64_t row = row0 + rr;
          if (row < m && j < c_hi) {
            load_row4<VEC>(G + row * n, j, n, g[u][rr]);
            load_row4<VEC>(E + row * n, j, n, e[u][rr]);
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) g[u][rr][q] = e[u][rr][q] = 0.0f;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kSubSteps; ++u) {
        const int jl = (s + u) * 128 + 4 * lane;  // column within the chunk
        const int64_t j = col0 + jl;
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
          const int64_t row = row0 + rr;
#pragma unroll
          for (int q = 0; q < 4; ++q) g[u][rr][q] = __fadd_rn(g[u][rr][q], e[u][rr][q]);
          if (row < m && j < c_hi) store_row4<VEC>(E + row * n, j, n, g[u][rr]);
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int c = 0; c < R; ++c)
              acc[rr][c] = fmaf(g[u][rr][q], qs[(jl + q) * R + c], acc[rr][c]);
        }
      }
    }
  }
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr)
#pragma unroll
    for (int c = 0; c < R; ++c) {
      float v = acc[rr][c];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      acc[rr][c] = v;
    }
  if (splits == 1) {
    if (lane == 0) {
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int64_t row = row0 + rr;
#pragma unroll
        for (int c = 0; c < R; ++c) {
          const float v = row < m ? acc[rr][c] : 0.0f;
          prow[warp * kRowsPerWarp + rr][c] = v;
          if (row < m) b.praw[row * R + c] = v;
        }
      }
    }
    __syncthreads();
  } else {
    // partial rows of this column range; the row range's last block adds
    // them in column-range order
    if (lane == 0) {
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int64_t row = row0 + rr;
        if (row >= m) continue;
#pragma unroll
        for (int c = 0; c < R; ++c) b.ppart[((int64_t)split * m + row) * R + c] = acc[rr][c];
      }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
      last = atomicAdd(&b.rb_tickets[blockIdx.x], 1u) == (uint32_t)splits - 1u;
    __syncthreads();
    if (!last) return;
    __threadfence();
    if (threadIdx.x < kRowsPerBlock * R) {
      const int rl = threadIdx.x / R, c = threadIdx.x % R;
      const int64_t row = (int64_t)blockIdx.x * kRowsPerBlock + rl;
      float v = 0.0f;
      if (row < m) {
        for (int sp = 0; sp < splits; ++sp) v += __ldcg(&b.ppart[((int64_t)sp * m + row) * R + c]);
        b.praw[row * R + c] = v;
      }
      prow[rl][c] = v;
    }
    if (threadIdx.x == 0) b.rb_tickets[blockIdx.x] = 0u;
    __syncthreads();
  }
  if (threadIdx.x < R * R) {
    const int a = threadIdx.x / R, c = threadIdx.x % R;
    double s = 0.0;
    for (int rr = 0; rr < kRowsPerBlock; ++rr) s += (double)prow[rr][a] * (double)prow[rr][c];
    b.gram_part[(int64_t)blockIdx.x * R * R + threadIdx.x] = s;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(&b.state->ticket_mq, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (threadIdx.x < R * R) {
    double s = 0.0;
    for (uint32_t blk = 0; blk < gridDim.x; ++blk)
      s += __ldcg(&b.gram_part[(int64_t)blk * R * R + threadIdx.x]);
    gram[threadIdx.x] = s;
  }
  __syncthreads();
  if (warp == 0) cholesky_inverse_warp<R>(gram, rinv, b.w, lane);
  if (threadIdx.x == 0) b.state->ticket_mq = 0u;
}

// ---------------------------------------------------------------------------
// pass 2: Q' = M^T P_hat with a deterministic split reduction.
// ---------------------------------------------------------------------------
template <int R, bool VEC>
__global__ void __launch_bounds__(kPThreads) psgd_mtp_kernel(
    const float* __restrict__ M, int64_t m, int64_t n, int64_t rows_per_split,
    int splits, float* __restrict__ P_out, float* __restrict__ Q_out, PsgdBufs b) {
  extern __shared__ float dyn[];
  float* ph = dyn;                                  // [kPhRows][R]
  float* red = dyn + kPhRows * R;                   // [kPWarps][kStrip][R]
  __shared__ float w[R * R];
  __shared__ bool last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int strip = blockIdx.x, split = blockIdx.y;
  const int64_t ra = (int64_t)split * rows_per_split;
  const int64_t rb = std::min<int64_t>(ra + rows_per_split, m);
  if (threadIdx.x < R * R) w[threadIdx.x] = b.w[threadIdx.x];
  const int64_t col = (int64_t)strip * kStrip + 4 * lane;
  float acc[4][R];
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int c = 0; c < R; ++c) acc[q][c] = 0.0f;
  for (int64_t sa = ra; sa < rb; sa += kPhRows) {
    const int64_t sb = std::min<int64_t>(sa + kPhRows, rb);
    __syncthreads();
    // P_hat = P W for rows [sa, sb) of this slice
    for (int64_t i = sa + threadIdx.x; i < sb; i += kPThreads) {
      float p[R];
#pragma unroll
      for (int a = 0; a < R; ++a) p[a] = b.praw[i * R + a];
#pragma unroll
      for (int c = 0; c < R; ++c) {
        float s = 0.0f;
#pragma unroll
        for (int a = 0; a <= c; ++a) s = fmaf(p[a], w[a * R + c], s);
        ph[(i - sa) * R + c] = s;
        if (strip == 0) P_out[i * R + c] = s;
      }
    }
    __syncthreads();
    if (col < n) {
      // four of the warp's rows loaded before their products
      for (int64_t i0 = sa + warp; i0 < sb; i0 += 4 * kPWarps) {
        float v[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t i = i0 + (int64_t)u * kPWarps;
          if (i < sb) {
            load_row4<VEC>(M + i * n, col, n, v[u]);
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) v[u][q] = 0.0f;
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t i = i0 + (int64_t)u * kPWarps;
          if (i >= sb) break;
          const float* pr = ph + (i - sa) * R;
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int c = 0; c < R; ++c) acc[q][c] = fmaf(v[u][q], pr[c], acc[q][c]);
        }
      }
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int c = 0; c < R; ++c) red[((int64_t)warp * kStrip + 4 * lane + q) * R + c] = acc[q][c];
  __syncthreads();
  for (int t = threadIdx.x; t < kStrip * R; t += kPThreads) {
    float s = 0.0f;
    for (int wv = 0; wv < kPWarps; ++wv) s += red[(int64_t)wv * kStrip * R + t];
    const int64_t c0 = (int64_t)strip * kStrip + t / R;
    if (c0 < n) b.q_part[((int64_t)split * n + c0) * R + (t % R)] = s;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(&b.tickets[strip], 1u) == (uint32_t)splits - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int t = threadIdx.x; t < kStrip * R; t += kPThreads) {
    const int64_t c0 = (int64_t)strip * kStrip + t / R;
    if (c0 >= n) continue;
    float s = 0.0f;
    for (int sp = 0; sp < splits; ++sp) s += __ldcg(&b.q_part[((int64_t)sp * n + c0) * R + (t % R)]);
    Q_out[c0 * R + (t % R)] = s;
  }
  if (threadIdx.x == 0) b.tickets[strip] = 0u;
}

// ---------------------------------------------------------------------------
// pass 3: E' = M - P_hat Q'^T.
// ---------------------------------------------------------------------------
template <int R, bool VEC>
__global__ void __launch_bounds__(kPThreads) psgd_residual_kernel(
    float* __restrict__ E, int64_t m, int64_t n, const float* __restrict__ P,
    const float* __restrict__ Q, int64_t cols_per_split) {
  __shared__ float qs[kQChunk * R];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t row0 = (int64_t)blockIdx.x * kRowsPerBlock + warp * kRowsPerWarp;
  const int64_t c_lo = (int64_t)blockIdx.y * cols_per_split;
  const int64_t c_hi = std::min<int64_t>(n, c_lo + cols_per_split);
  float p[kRowsPerWarp][R];
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr)
#pragma unroll
    for (int c = 0; c < R; ++c) p[rr][c] = (row0 + rr < m) ? P[(row0 + rr) * R + c] : 0.0f;
  for (int64_t col0 = c_lo; col0 < c_hi; col0 += kQChunk) {
    __syncthreads();
    stage_q<R>(qs, Q, col0, n);
    __syncthreads();
#pragma unroll
    for (int s = 0; s < kQChunk / 128; s += kSubSteps) {
      float v[kSubSteps][kRowsPerWarp][4];
#pragma unroll
      for (int u = 0; u < kSubSteps; ++u) {
        const int64_t j = col0 + (s + u) * 128 + 4 * lane;
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
          const int64_t row = row0 + rr;
          if (row < m && j < c_hi) {
            load_row4<VEC>(E + row * n, j, n, v[u][rr]);
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) v[u][rr][q] = 0.0f;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kSubSteps; ++u) {
        const int jl = (s + u) * 128 + 4 * lane;
        const int64_t j = col0 + jl;
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
          const int64_t row = row0 + rr;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float a = 0.0f;
#pragma unroll
            for (int c = 0; c < R; ++c) a = fmaf(p[rr][c], qs[(jl + q) * R + c], a);
            v[u][rr][q] = v[u][rr][q] - a;
          }
          if (row < m && j < c_hi) store_row4<VEC>(E + row * n, j, n, v[u][rr]);
        }
      }
    }
  }
}

// ===========================================================================
// Tensor-core path (n a multiple of 4, so that every row of G, E and M
// starts on a 16-byte boundary).
//
// Pass 1, P = M Q (K = n, N = r), runs as tcgen05.mma kind::tf32 with the
// accumulator (128 lanes of fp32) in tensor memory.  TF32 keeps 10 mantissa
// bits, so every operand is split as x = hi + lo (hi = x rounded to TF32,
// lo = x - hi exactly, of which the tensor core keeps the top 11 bits) and
// hi*hi + hi*lo + lo*hi is accumulated: about 2^-21 relative error per
// product instead of 2^-11, close to fp32.
//
// The memory system wants long runs of each matrix row (a pass that read
// 128 bytes of each of 128 rows per step reached 61 % of the bandwidth, the
// same pass reading 2 KB of each of 8 rows 89 %), while the MMA wants 128
// operand rows.  So an operand tile of 128 rows is made of SG segments of
// 32 columns from each of 128 / SG matrix rows, and the thin operand
// carries the segments along N: image row s r + c holds column c of Q for
// the segment s (rows SG r .. of hi, then as many of lo).  Operand row
// (row, s) times image row (s', c) is the segment-s part of P[row][c] when
// s' = s; the read-out keeps those and adds them over the segments.  SG = 4
// for r <= 4 (512 bytes of each of 32 rows per unit), 2 for r <= 8, 1
// above; the MMA work grows with SG (the off-diagonal products are wasted:
// 16 segments made the pass tensor-bound).
//
// Work: the pass cuts its K range into units of 32 SG columns per tile of
// 128 / SG rows; units are numbered tile-major and every CTA (one per SM)
// takes a contiguous run of them, so each CTA contributes a partial result
// to at most a few tiles.  CTA c's partial for tile t goes to slot c + t
// (the (CTA, tile) pairs, taken in unit order, advance one of the two at a
// time, so the slots are distinct), and the last contributor of a tile
// (ticket) adds the tile's slots in CTA order: deterministic.
//
// Roles in a CTA of 448 threads: warps 0-7 stream G and E (cp.async into
// staging slots of their own), form M = G + E (stored to global) and write
// hi(M), lo(M) into the swizzled operand stage; warp 8 lane 0 copies the Q
// images (bulk copies); warp 9 owns the tensor memory and its lane 0 issues
// the MMAs; warps 10-13 read the accumulator out (tcgen05.ld: warp w reads
// lanes 32 (w % 4) .. + 31) and do the per-tile reductions.  Operand
// stages are handed on by mbarriers: full (image landed), conv (operands
// written), empty (the MMAs reading the stage are done).  The accumulator
// is double-buffered (segment j in buffer j % 2; acc_full / acc_empty per
// buffer), so the converters never wait for a read-out: with one buffer
// and the read-out done by the converters, the pipeline drained at every
// segment end and the pass ran at about half the bandwidth on matrices of
// 4096 columns.  Every wait is bounded.  A converter warp gives up as one
// (a vote) and the converters share no barrier; the read-out warps take
// each abort decision together (a flag behind their named barrier), so no
// barrier is left waiting for a thread that gave up.
//
// Pass 2 (the column sums of M^T P, with W = U^-1 and P_hat = P W formed
// beside them; psgd_qfinal adds the sums and applies W) and pass 3 (E' =
// M - P_hat Q'^T) stream M on the CUDA cores; see their kernels.
// ===========================================================================
namespace tcp {
constexpr int kConv = 256;             // converter threads (warps 0-7)
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kEpiWarp0 = 10;          // accumulator read-out warps 10-13
constexpr int kEpi = 128;              // accumulator read-out threads
constexpr int kThreads = 448;
constexpr int kRows = 128;             // MMA M: operand rows of a tile
constexpr int kKBlk = 32;              // K per operand row of a unit (one 128-byte row)
constexpr uint32_t kTileBytes = kRows * kKBlk * 4;  // 16 KB
constexpr uint32_t kAccCols = 64;     // one accumulator buffer (3 H <= 64 columns)
constexpr uint32_t kTmemCols = 2 * kAccCols;
constexpr int kResidConv = 512;        // passes 2 and 3: compute threads (warps 0-15)
constexpr int kResidThreads = 544;     // passes 2 and 3: warps 0-15 compute, warp 16 loads
constexpr int kWThreads = 64;          // pass 2: warps 17-18 form W and P_hat
constexpr int kQThreads = kResidThreads + kWThreads;
constexpr int kGramSlots = 256;        // pass 2: partial Gram sums (max(kWThreads, r^2) doubles)
constexpr int kStagesR = 6;            // passes 2 and 3: stages (32 KB each)
constexpr long long kWaitCycles = 4000000000ll;  // bound on each wait: ~2 s at 2 GHz
constexpr int kPadRows = 16;           // P and P_hat rows are padded to a multiple of this

// Segments per operand tile for rank R (SG r <= 16: one 16-row image half).
__host__ __device__ constexpr int segs_for(int R) { return R <= 4 ? 4 : R <= 8 ? 2 : 1; }
// Image rows per half (hi or lo): SG r rounded up to 16.
__host__ __device__ constexpr int img_half(int R, int SG) { return (SG * R + 15) / 16 * 16; }
// Pass 1: operand stages (hi, lo and the image, 36 KB each) and staging
// slots of the converters' copies of G and E (32 KB each).
constexpr int kOpStages = 2;
constexpr int kStgSlots = 4;

// First unit of CTA c of C over U units, and the CTA that owns unit u: the
// largest c with floor(U c / C) <= u, i.e. U c < (u + 1) C.
__host__ __device__ __forceinline__ int64_t unit_lo(int c, int C, int64_t U) {
  return U * c / C;
}
__host__ __device__ __forceinline__ int unit_owner(int64_t u, int C, int64_t U) {
  return (int)(((u + 1) * C - 1) / U);
}

// Unit u of a tile-major numbering with `per` units per tile, stepped
// without a division per unit (64-bit division is a long instruction
// sequence on the GPU), and the stage ring position of the i-th unit of a
// run: stage st, parity ph of its use.
struct UnitCursor {
  int64_t tile, blk, per;
  __device__ __forceinline__ UnitCursor(int64_t u, int64_t per_)
      : tile(u / per_), blk(u % per_), per(per_) {}
  __device__ __forceinline__ void next() {
    if (++blk == per) {
      blk = 0;
      ++tile;
    }
  }
};
template <int S>
struct Ring {
  int st = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next() {
    if (++st == S) {
      st = 0;
      ph ^= 1u;
    }
  }
};

// Barrier of the read-out warps only.
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 2, %0;" ::"n"(kEpi) : "memory");
}
__device__ __forceinline__ void w_sync() {
  asm volatile("bar.sync 3, %0;" ::"n"(kWThreads) : "memory");
}

struct Smem {
  uint32_t a_hi;     // [S] operand tiles hi(M) (shared addresses)
  uint32_t a_lo;     // [S] operand tiles lo(M)
  uint32_t img;      // [S] thin-operand images
  uint32_t stg;      // [SS] staging slots of the converters' copies
  uint64_t* full;
  uint64_t* conv;
  uint64_t* empty;
  uint64_t* acc_full;   // [2] accumulator buffers
  uint64_t* acc_empty;  // [2]
  uint64_t* drain;
  uint32_t* tmem_slot;
  volatile int* epi_abort;   // the read-out warps' abort decision
  int* last1;
  int* last2;
  float* rows;   // [kRows][16]
  double* gram;  // [16 * 16]
};

__host__ __device__ constexpr size_t smem_bytes_p(int S, uint32_t img_bytes, int SS) {
  return 1024 + (size_t)S * (2 * kTileBytes + img_bytes) + (size_t)SS * 2 * kTileBytes +
         (size_t)(3 * S + 5) * 8 + 64 + (size_t)kRows * 16 * 4 + 16 * 16 * 8;
}

__device__ __forceinline__ Smem carve_smem(unsigned char* raw, int S, uint32_t img_bytes, int SS) {
  using namespace sm100;
  // the 128-byte swizzle repeats every 1024 bytes: tiles start on 1024
  unsigned char* p = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Smem s;
  s.a_hi = smem_u32(p); p += (size_t)S * kTileBytes;
  s.a_lo = smem_u32(p); p += (size_t)S * kTileBytes;
  s.img = smem_u32(p); p += (size_t)S * img_bytes;
  s.stg = smem_u32(p); p += (size_t)SS * 2 * kTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(p);
  s.full = bars;
  s.conv = bars + S;
  s.empty = bars + 2 * S;
  s.acc_full = bars + 3 * S;
  s.acc_empty = s.acc_full + 2;
  s.drain = s.acc_full + 4;
  p += (size_t)(3 * S + 5) * 8;
  s.tmem_slot = reinterpret_cast<uint32_t*>(p);
  s.epi_abort = reinterpret_cast<volatile int*>(p + 8);
  s.last1 = reinterpret_cast<int*>(p + 32);
  s.last2 = reinterpret_cast<int*>(p + 48);
  p += 64;
  s.rows = reinterpret_cast<float*>(p); p += (size_t)kRows * 16 * 4;
  s.gram = reinterpret_cast<double*>(p);
  return s;
}

// The read-out warps' common abort decision: any thread that saw a wait run
// out raises the flag, all read it after the group's named barrier.
__device__ __forceinline__ bool epi_abort_now(const Smem& s, bool ok) {
  if (!ok) *s.epi_abort = 1;
  epi_sync();
  return *s.epi_abort != 0;
}

struct TcBufs {
  float* praw;           // [m][R] P = M Q
  float* part;           // [(C + tiles)][rows of a tile][R] partials per (CTA, tile)
  float* qimg;           // [units along K][image] the Q images
  uint32_t* rt_tickets;  // [row tiles]
  double* gram_part;     // [row tiles][R][R]
  float* w;              // [R][R] U^-1
  PsgdState* state;
  uint32_t* status;
};

// ---------------------------------------------------------------------------
// pass 0: the images of Q for pass 1, one per 32 SG rows of Q (one thread
// per row of Q): row i = 32 SG kb + 32 s + k is column k of the image of
// block kb, where it fills rows s R + c (hi(Q[i][c])) and H + s R + c
// (lo), H = the half height; the threads of segment 0 also clear the
// padding rows.
// ---------------------------------------------------------------------------
template <int R, int SG>
__global__ void __launch_bounds__(256) psgd_qimage_kernel(const float* __restrict__ Q, int64_t n,
                                                          float* __restrict__ img, int64_t rows) {
  using namespace sm100;
  constexpr int H = img_half(R, SG);
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows) return;
  const int64_t kb = i / (kKBlk * SG);
  const uint32_t sgm = (uint32_t)((i / kKBlk) % SG), k = (uint32_t)(i % kKBlk);
  float* im = img + kb * (2 * H * kKBlk);
#pragma unroll
  for (int c = 0; c < R; ++c) {
    const float v = i < n ? Q[i * R + c] : 0.0f;
    const float h = to_tf32(v);
    im[sw128_offset(sgm * R + c, k) >> 2] = h;
    im[sw128_offset(H + sgm * R + c, k) >> 2] = v - h;
  }
  if (sgm == 0) {
    for (int row = SG * R; row < H; ++row) {
      im[sw128_offset(row, k) >> 2] = 0.0f;
      im[sw128_offset(H + row, k) >> 2] = 0.0f;
    }
  }
}

// ---------------------------------------------------------------------------
// pass 1 on the tensor cores: M = G + E (written over E) and P = M Q; the
// last contributor of a row tile adds its partial rows, writes the tile's
// P rows (zero-padded) and adds the tile's Gram matrix to its CTA's Gram
// partial, which every CTA writes at the end (pass 2 factors the sum).
//
// Each converter thread streams its own 16-byte pieces of G and E (four
// operand rows, one 16-byte column chunk) through a ring of SS staging
// slots with cp.async, SS - 1 units ahead, and reads back only its own
// pieces (no barrier for the staging); it then writes hi(M) and lo(M) into
// the swizzled operand stage the MMAs read, and M to global memory.  The
// loader warp only copies the Q images (bulk copies).
// ---------------------------------------------------------------------------
template <int R, int SG>
__global__ void __launch_bounds__(kThreads, 1) psgd_p_tc_kernel(
    const float* __restrict__ G, float* __restrict__ E, int64_t m, int64_t n, TcBufs b) {
  using namespace sm100;
  constexpr int RG = kRows / SG;                  // matrix rows per tile
  constexpr int KU = SG * kKBlk;                  // matrix columns per unit
  constexpr int H = img_half(R, SG);              // image rows per half
  constexpr uint32_t kImg = 2 * H * kKBlk * 4;    // image bytes
  constexpr int S = kOpStages, SS = kStgSlots;
  constexpr int kPasses = kRows * 8 / kConv;      // operand rows per converter thread
  extern __shared__ unsigned char tc_smem[];
  const Smem s = carve_smem(tc_smem, S, kImg, SS);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int C = gridDim.x, cta = blockIdx.x;
  const int64_t RT = (m + RG - 1) / RG, KB = (n + KU - 1) / KU, U = RT * KB;
  const int64_t m_pad = (m + kPadRows - 1) / kPadRows * kPadRows;
  const int64_t u0 = unit_lo(cta, C, U), u1 = unit_lo(cta + 1, C, U), nun = u1 - u0;
  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.conv[i], kConv);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.acc_full[i], 1);
      mbar_init(&s.acc_empty[i], kEpi);
    }
    mbar_init(s.drain, 1);
    *s.epi_abort = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(s.tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *s.tmem_slot;
  bool ok = true, mma_issued = false;
  int64_t loads = 0;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      UnitCursor cur(u0, KB);
      Ring<S> ring;
      for (int64_t i = 0; i < nun; ++i, cur.next(), ring.next()) {
        const int st = ring.st;
        if (i >= S && !mbar_wait(&s.empty[st], ring.ph ^ 1u, kWaitCycles)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&s.full[st], kImg);
        bulk_load_s(s.img + st * kImg, b.qimg + cur.blk * (kImg / 4), kImg, &s.full[st]);
        ++loads;
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      // per K = 8 step: A_hi x [B_hi | B_lo] into columns [0, 2H), A_lo x
      // B_hi into [2H, 3H)
      constexpr uint32_t id1 = idesc_tf32(kRows, 2 * H, 0), id2 = idesc_tf32(kRows, H, 0);
      int seg = 0;
      UnitCursor cur(u0, KB);
      Ring<S> ring;
      for (int64_t i = 0; i < nun; ++i, cur.next(), ring.next()) {
        const int st = ring.st;
        if (!mbar_wait(&s.conv[st], ring.ph, kWaitCycles) ||
            !mbar_wait(&s.full[st], ring.ph, kWaitCycles)) {
          ok = false;
          break;
        }
        const bool first = i == 0 || cur.blk == 0;
        // a segment accumulates into buffer seg & 1, free once the read-out
        // of segment seg - 2 is done
        const uint32_t d = tmem + (uint32_t)(seg & 1) * kAccCols;
        if (first && seg >= 2 &&
            !mbar_wait(&s.acc_empty[seg & 1], (uint32_t)(((seg - 2) >> 1) & 1), kWaitCycles)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t ah = s.a_hi + st * kTileBytes, al = s.a_lo + st * kTileBytes;
        const uint32_t im = s.img + st * kImg;
#pragma unroll
        for (int kk = 0; kk < kKBlk / 8; ++kk) {
          const uint32_t acc = (first && kk == 0) ? 0u : 1u;
          // operand rows of 128 bytes, 8-row groups 1024 bytes apart; a K = 8
          // step is 32 bytes along the rows
          const uint64_t db = smem_desc_sw128(im + kk * 32, 16, 1024);
          mma_tf32(d, smem_desc_sw128(ah + kk * 32, 16, 1024), db, id1, acc);
          mma_tf32(d + 2 * H, smem_desc_sw128(al + kk * 32, 16, 1024), db, id2, acc);
        }
        mma_issued = true;
        mma_commit(&s.empty[st]);
        if (cur.blk == KB - 1 || i == nun - 1) {
          mma_commit(&s.acc_full[seg & 1]);
          ++seg;
        }
      }
    }
  } else if (warp < kProducerWarp) {
    const uint32_t ch = lane & 7;
    // staging slot q holds piece j (0..3: G of operand row p = j, 4..7: E)
    // of thread t at stg + ((q * 8 + j) * kConv + t) * 16
    auto stage_unit = [&](int64_t rt, int64_t kb, int q) {
#pragma unroll
      for (int p = 0; p < kPasses; ++p) {
        const uint32_t a = p * (kConv / 8) + warp * 4 + (lane >> 3);
        const int64_t grow = rt * RG + a / SG;
        const int64_t col = kb * KU + (a % SG) * kKBlk + 4 * ch;
        const bool in = grow < m && col < n;  // n % 4 == 0: a chunk is in or out
        const int64_t off = in ? grow * n + col : 0;
        cp_async16_zfill(s.stg + ((q * 8 + p) * kConv + tid) * 16, G + off, in ? 16u : 0u);
        cp_async16_zfill(s.stg + ((q * 8 + 4 + p) * kConv + tid) * 16, E + off, in ? 16u : 0u);
      }
      cp_async_commit();
    };
    UnitCursor icur(u0, KB);
    for (int q = 0; q < SS - 1; ++q, icur.next()) {
      if (q < nun) stage_unit(icur.tile, icur.blk, q);
      else cp_async_commit();
    }
    UnitCursor cur(u0, KB);
    Ring<S> ring;
    int q = 0;  // staging slot of unit i
    for (int64_t i = 0; i < nun; ++i, cur.next(), ring.next(), icur.next(), q = (q + 1) % SS) {
      // unit i + SS - 1 goes into the slot unit i - 1 used
      if (i + SS - 1 < nun) stage_unit(icur.tile, icur.blk, (q + SS - 1) % SS);
      else cp_async_commit();
      cp_async_wait<SS - 1>();  // this thread's pieces of unit i have landed
      const int64_t rt = cur.tile, kb = cur.blk;
      float4 g[kPasses], e[kPasses];
#pragma unroll
      for (int p = 0; p < kPasses; ++p) {
        g[p] = lds128(s.stg + ((q * 8 + p) * kConv + tid) * 16);
        e[p] = lds128(s.stg + ((q * 8 + 4 + p) * kConv + tid) * 16);
      }
      float4 hi[kPasses], lo[kPasses];
#pragma unroll
      for (int p = 0; p < kPasses; ++p) {
        g[p] = make_float4(__fadd_rn(g[p].x, e[p].x), __fadd_rn(g[p].y, e[p].y),
                           __fadd_rn(g[p].z, e[p].z), __fadd_rn(g[p].w, e[p].w));
        hi[p] = make_float4(to_tf32(g[p].x), to_tf32(g[p].y), to_tf32(g[p].z), to_tf32(g[p].w));
        lo[p] = make_float4(g[p].x - hi[p].x, g[p].y - hi[p].y, g[p].z - hi[p].z,
                            g[p].w - hi[p].w);
      }
      // M to global memory: lanes 8q .. 8q + 7 write one 128-byte piece of a
      // matrix row, the warp's four operand rows being consecutive pieces
#pragma unroll
      for (int p = 0; p < kPasses; ++p) {
        const uint32_t a = p * (kConv / 8) + warp * 4 + (lane >> 3);
        const int64_t grow = rt * RG + a / SG;
        const int64_t col = kb * KU + (a % SG) * kKBlk + 4 * ch;
        if (grow < m && col < n) *reinterpret_cast<float4*>(E + grow * n + col) = g[p];
      }
      // the operand stage is free once the MMAs of unit i - S are done (a
      // warp gives up as one; no barrier of the converters follows, and the
      // other warps' own waits run out in turn)
      const int st = ring.st;
      const bool got = i < S || mbar_wait(&s.empty[st], ring.ph ^ 1u, kWaitCycles);
      if (__any_sync(0xffffffffu, !got)) { ok = false; break; }
      const uint32_t ah = s.a_hi + st * kTileBytes, al = s.a_lo + st * kTileBytes;
#pragma unroll
      for (int p = 0; p < kPasses; ++p) {
        const uint32_t a = p * (kConv / 8) + warp * 4 + (lane >> 3);
        const uint32_t off = sw128_offset(a, 4 * ch);
        sts128(ah + off, hi[p]);
        sts128(al + off, lo[p]);
      }
      fence_proxy_async_smem();
      mbar_arrive(&s.conv[st]);
    }
    cp_async_wait<0>();  // no copy of this thread may outlive the CTA
  } else {
    // read-out warps: warp w reads tensor-memory lanes 32 (w % 4) .. + 31,
    // lane = operand row (row / SG of the tile, segment row % SG).  Per
    // segment of this CTA (one per row tile it touches), in order: keep
    // image rows s R .. s R + R - 1 of each product, add the segments of a
    // row by shuffles (fixed order) and write the CTA's partial P rows.
    const int e = tid - kEpiWarp0 * 32;
    const uint32_t quarter = (uint32_t)warp & 3u, orow = quarter * 32 + lane;
    const uint32_t sgm = orow % SG, lo_col = sgm * R;
    // this CTA's Gram partial: the Gram matrices of the row tiles it
    // finishes, added in tile order (entry e + kEpi j in gacc[j])
    constexpr int kGE = (R * R + kEpi - 1) / kEpi;
    double gacc[kGE];
#pragma unroll
    for (int j = 0; j < kGE; ++j) gacc[j] = 0.0;
    const int64_t t_first = u0 / KB, t_last = nun > 0 ? (u1 - 1) / KB : t_first - 1;
    int seg = 0;
    for (int64_t rt = t_first; rt <= t_last; ++rt, ++seg) {
      const uint32_t buf = (uint32_t)(seg & 1);
      const bool got = mbar_wait(&s.acc_full[buf], (uint32_t)((seg >> 1) & 1), kWaitCycles);
      if (epi_abort_now(s, got)) { ok = false; break; }
      float prod[3][R];
#pragma unroll
      for (int x = 0; x < 3; ++x)
#pragma unroll
        for (int c = 0; c < R; ++c) prod[x][c] = 0.0f;
      tc_fence_after_sync();
      const uint32_t base = tmem + ((quarter * 32) << 16) + buf * kAccCols;
#pragma unroll
      for (int x = 0; x < 3; ++x) {
#pragma unroll
        for (int j = 0; j < H / 16; ++j) {
          float v[16];
          tmem_ld16(base + x * H + 16 * j, v);
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const uint32_t col = 16 * j + q;
#pragma unroll
            for (int c = 0; c < R; ++c)
              if (col == lo_col + c) prod[x][c] = v[q];
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive(&s.acc_empty[buf]);
      float v[R];
#pragma unroll
      for (int c = 0; c < R; ++c) {
        float t = (prod[0][c] + prod[1][c]) + prod[2][c];
#pragma unroll
        for (int o = SG / 2; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        v[c] = t;
      }
      if (sgm == 0) {
        float* dst = b.part + ((int64_t)(cta + rt) * RG + orow / SG) * R;
#pragma unroll
        for (int c = 0; c < R; ++c) dst[c] = v[c];
      }
      __threadfence();
      epi_sync();
      const int c_first = unit_owner(rt * KB, C, U), c_last = unit_owner(rt * KB + KB - 1, C, U);
      if (e == 0)
        *s.last1 = atomicAdd(&b.rt_tickets[rt], 1u) == (uint32_t)(c_last - c_first);
      epi_sync();
      if (!*s.last1) continue;
      __threadfence();
      // the row tile's P rows: partials added in CTA order (loads issued in
      // batches, the additions in order)
      if (e < RG) {
        const int64_t grow = rt * RG + e;
        constexpr int kB = R <= 4 ? 8 : R <= 8 ? 4 : 2;
        float pr[R];
#pragma unroll
        for (int c = 0; c < R; ++c) pr[c] = 0.0f;
        for (int c0 = c_first; c0 <= c_last; c0 += kB) {
          float v[kB][R];
#pragma unroll
          for (int j = 0; j < kB; ++j) {
            const float* src = b.part + ((int64_t)(c0 + j + rt) * RG + e) * R;
#pragma unroll
            for (int c = 0; c < R; ++c) v[j][c] = c0 + j <= c_last ? __ldcg(src + c) : 0.0f;
          }
#pragma unroll
          for (int j = 0; j < kB; ++j)
            if (c0 + j <= c_last) {
#pragma unroll
              for (int c = 0; c < R; ++c) pr[c] += v[j][c];
            }
        }
        // rows m .. m_pad - 1 of the padded P are zero
#pragma unroll
        for (int c = 0; c < R; ++c) {
          s.rows[e * 16 + c] = grow < m ? pr[c] : 0.0f;
          if (grow < m_pad) b.praw[grow * R + c] = grow < m ? pr[c] : 0.0f;
        }
      }
      if (e == 0) b.rt_tickets[rt] = 0u;
      epi_sync();
      // the tile's Gram matrix (fp64) into this CTA's partial
#pragma unroll
      for (int j = 0; j < kGE; ++j) {
        const int t = e + j * kEpi;
        if (t < R * R) {
          const int a = t / R, c = t % R;
          double acc2 = 0.0;
          for (int r = 0; r < RG; ++r)
            acc2 += (double)s.rows[r * 16 + a] * (double)s.rows[r * 16 + c];
          gacc[j] += acc2;
        }
      }
    }
    // every CTA writes its partial (zero if it finished no tile); pass 2
    // adds them in CTA order
#pragma unroll
    for (int j = 0; j < kGE; ++j) {
      const int t = e + j * kEpi;
      if (t < R * R) b.gram_part[(int64_t)cta * R * R + t] = gacc[j];
    }
  }
  // end: the loader waits for its copies still in flight, the MMA issuer
  // for its MMAs, then warp 9 frees the tensor memory
  if (warp == kProducerWarp && lane == 0) {
    for (int64_t j = std::max<int64_t>(0, loads - S); j < loads; ++j)
      if (!mbar_wait(&s.full[j % S], (uint32_t)((j / S) & 1), kWaitCycles))
        ok = false;
  }
  if (warp == kMmaWarp && lane == 0 && mma_issued) {
    mma_commit(s.drain);
    if (!mbar_wait(s.drain, 0, kWaitCycles)) ok = false;
  }
  if (!ok) atomicOr(b.status, kStatusWaitTimeout);
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// pass 3: E' = M - P_hat Q'^T, fp32 FMAs on the CUDA cores (r products per
// element).  The matrix streams in units of 16 rows x 512 columns (2 KB
// contiguous per row, two TMA boxes of 16 x 256 without swizzle) together
// with the unit's 16 rows of P_hat; units run column block by column block,
// so a thread keeps the Q' rows of its four columns in registers for as
// long as its CTA stays in one column block.
// ---------------------------------------------------------------------------
constexpr int kRGRows = 16;           // rows per unit
constexpr int kRGPer = kRGRows / 4;   // rows per thread (4 row phases)
constexpr int kRGCols = 512;          // columns per unit
constexpr uint32_t kRGTile = kRGRows * kRGCols * 4;  // 32 KB

// One unit row of P_hat (R floats, rows R * 4 bytes apart from a 128-byte
// aligned start) into registers: 16-byte loads when R is a multiple of 4
// (every row then starts on a 16-byte boundary), 8-byte loads when it is
// even, else one float at a time.
template <int R>
__device__ __forceinline__ void lds_prow(uint32_t a, float (&p)[R]) {
  if constexpr (R % 4 == 0) {
#pragma unroll
    for (int c = 0; c < R; c += 4) {
      const float4 v = sm100::lds128(a + c * 4);
      p[c] = v.x; p[c + 1] = v.y; p[c + 2] = v.z; p[c + 3] = v.w;
    }
  } else if constexpr (R % 2 == 0) {
#pragma unroll
    for (int c = 0; c < R; c += 2)
      sm100::lds64(a + c * 4, p[c], p[c + 1]);
  } else {
#pragma unroll
    for (int c = 0; c < R; ++c) p[c] = sm100::lds32(a + c * 4);
  }
}

template <int R>
__global__ void __launch_bounds__(kResidThreads, 1) psgd_resid_tma_kernel(
    const __grid_constant__ CUtensorMap tmE, float* __restrict__ E, int64_t m, int64_t n,
    const float* __restrict__ phat, const float* __restrict__ Qn, uint32_t* status) {
  using namespace sm100;
  constexpr int S = kStagesR;
  constexpr uint32_t kPBytes = kRGRows * R * 4;  // P_hat rows of one unit
  constexpr uint32_t kStageBytes = kRGTile + ((kPBytes + 127) / 128) * 128;
  constexpr int kLoader = kResidConv / 32;       // the loader warp
  extern __shared__ unsigned char tc_smem[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(tc_smem) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(base + (size_t)S * kStageBytes);
  uint64_t* empty = full + S;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + S);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int C = gridDim.x, cta = blockIdx.x;
  const int64_t RG = (m + kRGRows - 1) / kRGRows, CB = (n + kRGCols - 1) / kRGCols, U = RG * CB;
  const int64_t u0 = unit_lo(cta, C, U), u1 = unit_lo(cta + 1, C, U);
  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kResidConv / 32);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  bool ok = true;
  int64_t loads = 0;
  if (warp == kLoader) {
    if (lane == 0) {
      tma_prefetch_map(&tmE);
      UnitCursor cur(u0, RG);
      Ring<S> ring;
      for (int64_t i = 0; i < u1 - u0; ++i, cur.next(), ring.next()) {
        const int st = ring.st;
        if (i >= S && !mbar_wait(&empty[st], ring.ph ^ 1u, kWaitCycles)) {
          ok = false;
          break;
        }
        // the warps read the stage through the generic proxy and the refill
        // writes it through the asynchronous one: order those reads (made
        // visible to this thread by the barrier) before the copy
        fence_proxy_async_smem();
        const int64_t cb = cur.tile, rg = cur.blk;
        unsigned char* stage = base + (size_t)st * kStageBytes;
        mbar_arrive_expect_tx(&full[st], kRGTile + kPBytes);
        tma_load_2d(stage, &tmE, (int32_t)(cb * kRGCols), (int32_t)(rg * kRGRows), &full[st]);
        tma_load_2d(stage + kRGTile / 2, &tmE, (int32_t)(cb * kRGCols + kRGCols / 2),
                    (int32_t)(rg * kRGRows), &full[st]);
        bulk_load(stage + kRGTile, phat + rg * kRGRows * R, kPBytes, &full[st]);
        ++loads;
      }
      for (int64_t j = std::max<int64_t>(0, loads - S); j < loads; ++j)
        if (!mbar_wait(&full[j % S], (uint32_t)((j / S) & 1), kWaitCycles))
          ok = false;
    }
  } else {
    // thread t: column chunk t % 128 (four columns), rows t / 128 + 4 h
    const uint32_t chunk = tid & 127, r0 = tid >> 7;
    int64_t cur_cb = -1;
    float qv[4][R];
    UnitCursor cur(u0, RG);
    Ring<S> ring;
    for (int64_t i = 0; i < u1 - u0; ++i, cur.next(), ring.next()) {
      const int st = ring.st;
      const int64_t cb = cur.tile, rg = cur.blk;
      const int64_t col = cb * kRGCols + 4 * chunk;
      if (cb != cur_cb) {
        // Q' rows of this thread's four columns for the new column block
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int c = 0; c < R; ++c) qv[q][c] = (col + q < n) ? __ldg(&Qn[(col + q) * R + c]) : 0.0f;
        cur_cb = cb;
      }
      // a wait that runs out ends the warp's loop (the warp decides as one,
      // as it meets at __syncwarp below; no other barrier follows)
      bool bad = *abort_flag != 0 || !mbar_wait(&full[st], ring.ph, kWaitCycles);
      if (__any_sync(0xffffffffu, bad)) {
        *abort_flag = 1;
        ok = false;
        break;
      }
      const uint32_t t = smem_u32(base + (size_t)st * kStageBytes);
      const uint32_t ps = t + kRGTile;
      // box (chunk / 64) holds columns 256 (chunk / 64) ..; rows 1 KB apart
      const uint32_t cofs = (chunk >> 6) * (kRGTile / 2) + (chunk & 63) * 16;
      float4 mv[kRGPer];
      float pr[kRGPer][R];
#pragma unroll
      for (int h = 0; h < kRGPer; ++h) {
        const uint32_t row = r0 + 4 * h;
        mv[h] = lds128(t + cofs + row * 1024);
        lds_prow<R>(ps + row * R * 4, pr[h]);
      }
      float4 out[kRGPer];
#pragma unroll
      for (int h = 0; h < kRGPer; ++h) {
        float x[4] = {mv[h].x, mv[h].y, mv[h].z, mv[h].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float a = 0.0f;
#pragma unroll
          for (int c = 0; c < R; ++c) a = fmaf(pr[h][c], qv[q][c], a);
          x[q] = x[q] - a;
        }
        out[h] = make_float4(x[0], x[1], x[2], x[3]);
      }
      // the stage can be refilled once every warp has read it: each lane's
      // results are computed here, so its loads from the stage have
      // returned, before the warp's one arrival
#pragma unroll
      for (int h = 0; h < kRGPer; ++h) settle(out[h]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
#pragma unroll
      for (int h = 0; h < kRGPer; ++h) {
        const int64_t grow = rg * kRGRows + r0 + 4 * h;
        if (grow < m && col < n) *reinterpret_cast<float4*>(E + grow * n + col) = out[h];
      }
    }
  }
  if (!ok) atomicOr(status, kStatusWaitTimeout);
  __syncthreads();
}

// ---------------------------------------------------------------------------
// pass 2: M^T P, fp32 FMAs on the CUDA cores (r products per element); the
// final reduction and Q' = (M^T P) W follow in psgd_qfinal, W and P_hat are
// formed here by two extra warps.  The tensor core cannot take this
// contraction's operand from M
// as it lies in memory: the sum runs over M's rows, so M would be the
// transposed (MN-major) operand, which kind::tf32 does not accept (it reads
// as zero), and transposing every tile through shared memory, plus one
// M = 128 MMA per 4 KB of M, held a tensor-core version of this pass near a
// third of the memory bandwidth.  Here M streams exactly as in pass 3 (units
// of 16 rows x 512 columns, column block by column block, with the unit's
// rows of P), and each thread keeps the sums of four columns in registers
// while its CTA stays in one column block.  Thread t holds columns
// 4 (t / 4) .. + 3 of rows t % 4 + 4 h of each unit; at the end of a column
// block the four row phases are added by shuffles (fixed order) and each
// CTA writes its partial sums of the block to slot CTA + block.
// ---------------------------------------------------------------------------
template <int R>
__global__ void __launch_bounds__(kQThreads, 1) psgd_qstream_kernel(
    const __grid_constant__ CUtensorMap tmM, int64_t m, int64_t n, const float* __restrict__ pp,
    const double* __restrict__ gram_part, int64_t gram_parts, float* __restrict__ P_out,
    float* __restrict__ phat, float* __restrict__ w_out, float* __restrict__ part,
    uint32_t* status) {
  using namespace sm100;
  constexpr int S = kStagesR;
  constexpr uint32_t kPBytes = kRGRows * R * 4;
  constexpr uint32_t kStageBytes = kRGTile + ((kPBytes + 127) / 128) * 128;
  constexpr int kLoader = kResidConv / 32;
  constexpr int R2 = R * R;
  extern __shared__ unsigned char tc_smem[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(tc_smem) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(base + (size_t)S * kStageBytes);
  uint64_t* empty = full + S;
  uint64_t* wbar = empty + S;  // (space kept: flags and the W work area follow)
  volatile int* abort_flag = reinterpret_cast<volatile int*>(wbar + 1);
  double* sg = reinterpret_cast<double*>(wbar + 2);  // [threads per entry][R2] partial Gram sums
  double* sgram = sg + kGramSlots;                    // [R2]
  float* sw = reinterpret_cast<float*>(sgram + 256);  // [R2] W
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int C = gridDim.x, cta = blockIdx.x;
  const int64_t RG = (m + kRGRows - 1) / kRGRows, CB = (n + kRGCols - 1) / kRGCols, U = RG * CB;
  const int64_t u0 = unit_lo(cta, C, U), u1 = unit_lo(cta + 1, C, U);
  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kResidConv / 32);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  bool ok = true;
  int64_t loads = 0;
  if (warp > kLoader) {
    // W = U^-1, U the Cholesky factor of P^T P, from the pass-1 Gram
    // partials (one per pass-1 CTA, added in the same fixed order in every
    // CTA), while the other warps
    // stream M; then this CTA's slice of P_hat = P W.
    const int wt = tid - (kLoader + 1) * 32;
    constexpr int HS = R2 >= kWThreads ? 1 : kWThreads / R2;  // threads per Gram entry
    for (int j = wt; j < R2 * HS; j += kWThreads) {
      const int t = j % R2, h = j / R2;
      double acc2 = 0.0;
      int64_t r = h;
      for (; r + 7 * HS < gram_parts; r += 8 * HS) {
        double v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = __ldcg(&gram_part[(r + q * HS) * R2 + t]);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc2 += v[q];
      }
      for (; r < gram_parts; r += HS) acc2 += __ldcg(&gram_part[r * R2 + t]);
      sg[h * R2 + t] = acc2;
    }
    w_sync();
    for (int t = wt; t < R2; t += kWThreads) {
      double a = 0.0;
      for (int h = 0; h < HS; ++h) a += sg[h * R2 + t];
      sgram[t] = a;
    }
    w_sync();
    if (wt < 32) {
      cholesky_inverse_warp<R>(sgram, sg, sw, lane);  // (sg is free again: rinv)
      if (lane == 0 && cta == 0)
        for (int t = 0; t < R2; ++t) w_out[t] = sw[t];  // for the Q' reduction
    }
    w_sync();
    const int64_t m_pad = RG * kRGRows;
    const int64_t ra = m_pad * cta / C, rb = m_pad * (cta + 1) / C;
    for (int64_t row = ra + wt; row < rb; row += kWThreads) {
      float pr[R];
#pragma unroll
      for (int a = 0; a < R; ++a) pr[a] = pp[row * R + a];
#pragma unroll
      for (int c = 0; c < R; ++c) {
        float acc = 0.0f;
#pragma unroll
        for (int a = 0; a <= c; ++a) acc = fmaf(pr[a], sw[a * R + c], acc);
        phat[row * R + c] = acc;
        if (row < m) P_out[row * R + c] = acc;
      }
    }
  } else if (warp == kLoader) {
    if (lane == 0) {
      tma_prefetch_map(&tmM);
      UnitCursor cur(u0, RG);
      Ring<S> ring;
      for (int64_t i = 0; i < u1 - u0; ++i, cur.next(), ring.next()) {
        const int st = ring.st;
        if (i >= S && !mbar_wait(&empty[st], ring.ph ^ 1u, kWaitCycles)) {
          ok = false;
          break;
        }
        // the warps read the stage through the generic proxy and the refill
        // writes it through the asynchronous one: order those reads (made
        // visible to this thread by the barrier) before the copy
        fence_proxy_async_smem();
        const int64_t cb = cur.tile, rg = cur.blk;
        unsigned char* stage = base + (size_t)st * kStageBytes;
        mbar_arrive_expect_tx(&full[st], kRGTile + kPBytes);
        tma_load_2d(stage, &tmM, (int32_t)(cb * kRGCols), (int32_t)(rg * kRGRows), &full[st]);
        tma_load_2d(stage + kRGTile / 2, &tmM, (int32_t)(cb * kRGCols + kRGCols / 2),
                    (int32_t)(rg * kRGRows), &full[st]);
        bulk_load(stage + kRGTile, pp + rg * kRGRows * R, kPBytes, &full[st]);
        ++loads;
      }
      for (int64_t j = std::max<int64_t>(0, loads - S); j < loads; ++j)
        if (!mbar_wait(&full[j % S], (uint32_t)((j / S) & 1), kWaitCycles))
          ok = false;
    }
  } else {
    // ranks up to 8: thread t takes four columns (chunk t / 4) and rows
    // t % 4 + 4 h of a unit; above 8, two columns (chunk t / 2) and rows
    // t % 2 + 2 h, so that the accumulators (columns x R) stay in registers
    constexpr int NC = R <= 8 ? 4 : 2;    // columns per thread
    constexpr int RP = NC == 4 ? 4 : 2;   // row phases
    constexpr int NH = kRGRows / RP;      // rows per thread and unit
    const uint32_t r0 = tid % RP, chunk = tid / RP;
    // chunks of NC columns; box (chunk / (256 / NC)) holds columns 256 (chunk / (256 / NC)) ..
    constexpr uint32_t kPerBox = 256 / NC;
    const uint32_t cofs = (chunk / kPerBox) * (kRGTile / 2) + (chunk % kPerBox) * (4 * NC);
    float acc[NC][R];
#pragma unroll
    for (int q = 0; q < NC; ++q)
#pragma unroll
      for (int c = 0; c < R; ++c) acc[q][c] = 0.0f;
    UnitCursor cur(u0, RG);
    Ring<S> ring;
    for (int64_t i = 0; i < u1 - u0; ++i, cur.next(), ring.next()) {
      const int st = ring.st;
      const int64_t cb = cur.tile;
      // a wait that runs out makes the warp (deciding as one) skip its work
      // from then on; it still meets the barriers at the ends of column blocks
      bool bad = *abort_flag != 0;
      if (!bad) bad = !mbar_wait(&full[st], ring.ph, kWaitCycles);
      const bool skip = __any_sync(0xffffffffu, bad);
      if (skip) {
        *abort_flag = 1;
        ok = false;
      }
      const uint32_t t = smem_u32(base + (size_t)st * kStageBytes);
      const uint32_t ps = t + kRGTile;
      // rows one after the other (ranks above 8 keep one row's P in
      // registers at a time)
      constexpr int kHU = R <= 8 ? NH : 1;
#pragma unroll kHU
      for (int h = 0; h < NH; ++h) {
        const uint32_t row = r0 + RP * h;
        float x[NC];
#pragma unroll
        for (int q = 0; q < NC; ++q) x[q] = 0.0f;
        float pr[R];
#pragma unroll
        for (int c = 0; c < R; ++c) pr[c] = 0.0f;
        if (!skip) {
          if constexpr (NC == 4) {
            const float4 mv = lds128(t + cofs + row * 1024);
            x[0] = mv.x; x[1] = mv.y; x[2] = mv.z; x[3] = mv.w;
          } else {
            lds64(t + cofs + row * 1024, x[0], x[1]);
          }
          lds_prow<R>(ps + row * R * 4, pr);
        }
#pragma unroll
        for (int q = 0; q < NC; ++q)
#pragma unroll
          for (int c = 0; c < R; ++c) acc[q][c] = fmaf(x[q], pr[c], acc[q][c]);
      }
      if (!skip) {
        // the stage can be refilled once every warp has read it: each lane's
        // sums are brought up to date here, so its loads from the stage
        // have returned, before the warp's one arrival
#pragma unroll
        for (int q = 0; q < NC; ++q)
#pragma unroll
          for (int c = 0; c < R; ++c) settle(acc[q][c]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
      if (cur.blk != RG - 1 && i != u1 - u0 - 1) continue;
      // end of this CTA's part of column block cb: its partial sums (the
      // row phases are adjacent lanes)
#pragma unroll
      for (int q = 0; q < NC; ++q)
#pragma unroll
        for (int c = 0; c < R; ++c) {
          float v = acc[q][c];
#pragma unroll
          for (int o = 1; o < RP; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          acc[q][c] = v;
        }
      if (r0 == 0) {
        float* dst = part + ((int64_t)(cta + cb) * kRGCols + NC * chunk) * R;
#pragma unroll
        for (int q = 0; q < NC; ++q)
#pragma unroll
          for (int c = 0; c < R; ++c) dst[q * R + c] = acc[q][c];
      }
#pragma unroll
      for (int q = 0; q < NC; ++q)
#pragma unroll
        for (int c = 0; c < R; ++c) acc[q][c] = 0.0f;
    }
  }
  if (!ok) atomicOr(status, kStatusWaitTimeout);
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Q' = (M^T P) W from pass 2's partial column sums (slot c + b holds CTA c's
// sums over its rows of column block b).  Block (b, x) takes 64 columns of
// column block b: four threads per column add every fourth of the block's
// contributing slots in CTA order, the four sums are added in a fixed order
// and W is applied.  As a grid of its own the reduction runs on every SM
// at once; done by the last contributor of each block inside pass 2 it
// formed a tail of about 9 us after the stream.
// ---------------------------------------------------------------------------
constexpr int kQFCols = 64;  // columns per block
template <int R>
__global__ void __launch_bounds__(256) psgd_qfinal_kernel(const float* __restrict__ part,
                                                          int64_t m, int64_t n, int C,
                                                          const float* __restrict__ W,
                                                          float* __restrict__ Q_out) {
  __shared__ float red[4][kQFCols][R];
  __shared__ float w[R * R];
  constexpr int kSub = kRGCols / kQFCols;
  const int64_t RG = (m + kRGRows - 1) / kRGRows, CB = (n + kRGCols - 1) / kRGCols, U = RG * CB;
  const int64_t cb = blockIdx.x / kSub;
  const int cl = threadIdx.x % kQFCols, qt = threadIdx.x / kQFCols;
  const int64_t lc = (int64_t)(blockIdx.x % kSub) * kQFCols + cl;  // column within the block
  const int64_t col = cb * kRGCols + lc;
  for (int t = threadIdx.x; t < R * R; t += blockDim.x) w[t] = W[t];
  const int c_first = unit_owner(cb * RG, C, U), c_last = unit_owner(cb * RG + RG - 1, C, U);
  float q[R];
#pragma unroll
  for (int c = 0; c < R; ++c) q[c] = 0.0f;
  if (col < n) {
    constexpr int kB = R <= 4 ? 8 : R <= 8 ? 4 : 2;
    for (int c0 = c_first + qt; c0 <= c_last; c0 += 4 * kB) {
      float v[kB][R];
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        const int cc = c0 + 4 * j;
        const float* src = part + ((int64_t)(cc + cb) * kRGCols + lc) * R;
#pragma unroll
        for (int c = 0; c < R; ++c) v[j][c] = cc <= c_last ? __ldcg(src + c) : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < kB; ++j)
        if (c0 + 4 * j <= c_last) {
#pragma unroll
          for (int c = 0; c < R; ++c) q[c] += v[j][c];
        }
    }
  }
#pragma unroll
  for (int c = 0; c < R; ++c) red[qt][cl][c] = q[c];
  __syncthreads();
  if (qt == 0 && col < n) {
    float t[R];
#pragma unroll
    for (int c = 0; c < R; ++c)
      t[c] = ((red[0][cl][c] + red[1][cl][c]) + red[2][cl][c]) + red[3][cl][c];
#pragma unroll
    for (int c = 0; c < R; ++c) {
      float acc = 0.0f;
#pragma unroll
      for (int a = 0; a <= c; ++a) acc = fmaf(t[a], w[a * R + c], acc);
      Q_out[col * R + c] = acc;
    }
  }
}

template <int R>
__host__ constexpr size_t resid_smem_bytes() {
  return 1024 + (size_t)kStagesR * (kRGTile + ((kRGRows * R * 4 + 127) / 128) * 128) +
         (size_t)2 * kStagesR * 8 + 16;
}
// pass 2 adds W's barrier, the Gram partial sums, the Gram matrix and W
template <int R>
__host__ constexpr size_t qstream_smem_bytes() {
  return resid_smem_bytes<R>() + 16 + (size_t)(kGramSlots + 256) * 8 + 256 * 4;
}

}  // namespace tcp

// cuTensorMapEncodeTiled from the driver (looked up once).
PFN_cuTensorMapEncodeTiled_v12000 encode_tiled_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// A rows x cols fp32 row-major matrix (cols a multiple of 4) read in boxes
// of box_rows x box_cols, with the 128-byte swizzle (box_cols <= 32) or
// rows stored one after the other; out-of-range parts of a box read as
// zero.
bool make_map(CUtensorMap* map, const float* base, int64_t rows, int64_t cols, uint32_t box_cols,
              uint32_t box_rows, bool swizzle) {
  const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Bytes of the tensor-core path's data area for matrices up to max_m x
// max_n: pass 1 partials and Q images, pass 2 partials, P and P_hat padded.
int64_t tc_area_bytes(int64_t max_m, int64_t max_n, int max_r, int num_sms) {
  auto up = [](int64_t b) { return (b + 255) / 256 * 256; };
  return up((int64_t)sizeof(float) * ((int64_t)num_sms * tcp::kRows + max_m + tcp::kRows) *
            max_r) +
         up(round_up(max_n, 512) * 128 + 16384) +
         up((int64_t)sizeof(float) * (num_sms + ceil_div(max_n, tcp::kRGCols)) * tcp::kRGCols *
            max_r) +
         2 * up((int64_t)sizeof(float) * round_up(max_m, tcp::kPadRows) * max_r);
}

// Pass 0 and pass 1 with SG segments per operand tile.
template <int R, int SG>
gc_status launch_pass1(gc_ctx* ctx, const float* grad, float* err, int64_t m, int64_t n,
                       const float* Q, const tcp::TcBufs& b) {
  constexpr int RG = tcp::kRows / SG, KU = SG * tcp::kKBlk, H = tcp::img_half(R, SG);
  constexpr uint32_t kImg = 2 * H * tcp::kKBlk * 4;
  const int64_t KB = ceil_div(n, KU), U = ceil_div(m, RG) * KB;
  const size_t smem = tcp::smem_bytes_p(tcp::kOpStages, kImg, tcp::kStgSlots);
  if (cudaFuncSetAttribute(tcp::psgd_p_tc_kernel<R, SG>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return GC_ERR_CUDA;
  {
    LaunchScope L(ctx, GC_PHASE_PSGD_THIN);
    const int64_t rows = KB * KU;
    tcp::psgd_qimage_kernel<R, SG><<<(unsigned)ceil_div(rows, 256), 256, 0, ctx->stream>>>(
        Q, n, b.qimg, rows);
  }
  {
    LaunchScope L(ctx, GC_PHASE_PSGD_MQ);
    const int c1 = (int)std::min<int64_t>(ctx->num_sms, U);
    tcp::psgd_p_tc_kernel<R, SG><<<c1, tcp::kThreads, smem, ctx->stream>>>(grad, err, m, n, b);
  }
  return GC_OK;
}

template <int R>
gc_status run_psgd_tc(gc_ctx* ctx, const float* grad, float* err, int64_t m, int64_t n,
                      float* P_out, float* Q_inout, const PsgdBufs& pb, char* area) {
  cudaStream_t s = ctx->stream;
  const PsgdWorkspace& pw = ctx->psgd;
  auto up = [](int64_t v) { return (v + 255) / 256 * 256; };
  tcp::TcBufs b;
  b.part = reinterpret_cast<float*>(area);
  area += up((int64_t)sizeof(float) * ((int64_t)ctx->num_sms * tcp::kRows + pw.max_m + tcp::kRows) *
             pw.max_r);
  b.qimg = reinterpret_cast<float*>(area);
  area += up(round_up(pw.max_n, 512) * 128 + 16384);
  float* qpart = reinterpret_cast<float*>(area);
  area += up((int64_t)sizeof(float) * (ctx->num_sms + ceil_div(pw.max_n, tcp::kRGCols)) *
             tcp::kRGCols * pw.max_r);
  const int64_t pad_bytes = up((int64_t)sizeof(float) * round_up(pw.max_m, tcp::kPadRows) * pw.max_r);
  b.praw = reinterpret_cast<float*>(area);  // P, rows padded with zeros to a multiple of 16
  area += pad_bytes;
  float* phat = reinterpret_cast<float*>(area);  // P_hat, padded the same way
  b.rt_tickets = pb.rb_tickets;
  b.gram_part = pb.gram_part;
  b.w = pb.w;
  b.state = pb.state;
  b.status = pb.status;

  const gc_status st1 = launch_pass1<R, tcp::segs_for(R)>(ctx, grad, err, m, n, Q_inout, b);
  if (st1 != GC_OK) return st1;

  // passes 2 and 3 stream M in units of 16 rows x 512 columns; pass 2 also
  // forms W and P_hat = P W
  CUtensorMap tm_r;
  if (!make_map(&tm_r, err, m, n, tcp::kRGCols / 2, tcp::kRGRows, false)) return GC_ERR_CUDA;
  const int64_t m_pad = round_up(m, tcp::kRGRows);
  const int c3 = (int)std::min<int64_t>(ctx->num_sms,
                                        (m_pad / tcp::kRGRows) * ceil_div(n, tcp::kRGCols));
  const size_t sm2 = tcp::qstream_smem_bytes<R>(), sm3 = tcp::resid_smem_bytes<R>();
  if (cudaFuncSetAttribute(tcp::psgd_qstream_kernel<R>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2) != cudaSuccess ||
      cudaFuncSetAttribute(tcp::psgd_resid_tma_kernel<R>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3) != cudaSuccess)
    return GC_ERR_CUDA;
  {
    LaunchScope L(ctx, GC_PHASE_PSGD_MTP);
    // one Gram partial per pass-1 CTA
    const int64_t gram_parts = std::min<int64_t>(
        ctx->num_sms,
        ceil_div(m, tcp::kRows / tcp::segs_for(R)) * ceil_div(n, tcp::segs_for(R) * tcp::kKBlk));
    tcp::psgd_qstream_kernel<R><<<c3, tcp::kQThreads, sm2, s>>>(
        tm_r, m, n, b.praw, b.gram_part, gram_parts, P_out, phat, b.w, qpart, b.status);
  }
  {
    LaunchScope L(ctx, GC_PHASE_PSGD_THIN);
    const int64_t blocks = ceil_div(n, tcp::kRGCols) * (tcp::kRGCols / tcp::kQFCols);
    tcp::psgd_qfinal_kernel<R><<<(unsigned)blocks, 256, 0, s>>>(qpart, m, n, c3, b.w, Q_inout);
  }
  {
    LaunchScope L(ctx, GC_PHASE_PSGD_RESID);
    tcp::psgd_resid_tma_kernel<R><<<c3, tcp::kResidThreads, sm3, s>>>(tm_r, err, m, n, phat,
                                                                        Q_inout, b.status);
  }
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

// Gram partials the workspace holds: the CUDA-core path writes one per
// block of 8 rows, the tensor-core path one per pass-1 CTA (at most one per SM).
int64_t gram_parts_cap(int64_t max_m, int num_sms) {
  return std::max<int64_t>(ceil_div(max_m, 8), num_sms);
}

template <int R, bool VEC>
gc_status run_psgd(gc_ctx* ctx, const float* grad, float* err, int64_t m, int64_t n,
                   float* P_out, float* Q_inout) {
  cudaStream_t s = ctx->stream;
  const PsgdWorkspace& pw = ctx->psgd;
  char* base = static_cast<char*>(ctx->psgd_base);
  PsgdBufs b;
  // carve the reserved scratch (see gc_ctx_reserve_powersgd)
  size_t off = 0;
  auto take = [&](size_t bytes) { void* p = base + off; off += (bytes + 255) / 256 * 256; return p; };
  // tickets and state first (zero between calls, shared by both paths),
  // then the data both paths write before they read
  b.state = static_cast<PsgdState*>(take(sizeof(PsgdState)));
  b.w = static_cast<float*>(take(sizeof(float) * 16 * 16));
  b.tickets = static_cast<uint32_t*>(take(sizeof(uint32_t) * ceil_div(pw.max_n, kStrip)));
  // (row tickets: one per 8 rows covers both paths; Gram partials: one per
  // 8 rows or per SM, whichever is more)
  b.rb_tickets = static_cast<uint32_t*>(take(sizeof(uint32_t) * ceil_div(pw.max_m, 8)));
  b.praw = static_cast<float*>(take(sizeof(float) * pw.max_m * pw.max_r));
  b.gram_part = static_cast<double*>(
      take(sizeof(double) * gram_parts_cap(pw.max_m, ctx->num_sms) * pw.max_r * pw.max_r));
  b.status = ctx->ws.status;
  if constexpr (VEC) {
    // rows start on 16-byte boundaries: the tensor-core path
    return run_psgd_tc<R>(ctx, grad, err, m, n, P_out, Q_inout, b, base + off);
  }
  b.ppart = static_cast<float*>(take(sizeof(float) * kMaxColSplits * pw.max_m * pw.max_r));
  b.q_part = reinterpret_cast<float*>(base + off);
  const int64_t qcap = (pw.bytes - (int64_t)off) / (int64_t)sizeof(float);

  const int mq_blocks = (int)ceil_div(m, kRowsPerBlock);
  // column ranges (multiples of kQChunk) so that passes 1 and 3 have about
  // 8 blocks per SM
  const int64_t chunks = ceil_div(n, kQChunk);
  int64_t csplits = std::min<int64_t>(
      {(int64_t)kMaxColSplits, chunks, std::max<int64_t>(1, ceil_div((int64_t)ctx->num_sms * 8, mq_blocks))});
  const int64_t cps = ceil_div(chunks, csplits) * kQChunk;
  csplits = ceil_div(n, cps);
  {
    LaunchScope L(ctx, GC_PHASE_PSGD_MQ);
    psgd_mq_kernel<R, VEC><<<dim3(mq_blocks, (unsigned)csplits), kPThreads, 0, s>>>(
        grad, err, m, n, Q_inout, b, cps);
  }

  const int strips = (int)ceil_div(n, kStrip);
  int64_t splits = std::max<int64_t>(1, ceil_div((int64_t)ctx->num_sms * 4, strips));
  splits = std::min<int64_t>(splits, std::max<int64_t>(1, ceil_div(m, 32)));
  splits = std::min<int64_t>(splits, std::max<int64_t>(1, qcap / (n * R)));
  const int64_t rows_per_split = ceil_div(m, splits);
  splits = ceil_div(m, rows_per_split);
  const size_t smem = sizeof(float) * ((int64_t)kPhRows * R + (int64_t)kPWarps * kStrip * R);
  // dynamic + static shared memory above the 48 KB default needs an opt-in
  if (smem + sizeof(float) * R * R + 64 > 48 * 1024) {
    if (cudaFuncSetAttribute(psgd_mtp_kernel<R, VEC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return GC_ERR_CUDA;
  }
  {
    LaunchScope L(ctx, GC_PHASE_PSGD_MTP);
    psgd_mtp_kernel<R, VEC><<<dim3(strips, (unsigned)splits), kPThreads, smem, s>>>(
        err, m, n, rows_per_split, (int)splits, P_out, Q_inout, b);
  }
  {
    LaunchScope L(ctx, GC_PHASE_PSGD_RESID);
    psgd_residual_kernel<R, VEC><<<dim3(mq_blocks, (unsigned)csplits), kPThreads, 0, s>>>(
        err, m, n, P_out, Q_inout, cps);
  }
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

template <int R>
gc_status run_psgd_r(gc_ctx* ctx, const float* grad, float* err, int64_t m, int64_t n,
                     float* P_out, float* Q_inout) {
  if (n % 4 == 0) return run_psgd<R, true>(ctx, grad, err, m, n, P_out, Q_inout);
  return run_psgd<R, false>(ctx, grad, err, m, n, P_out, Q_inout);
}

}  // namespace

int64_t psgd_workspace_bytes(int64_t max_m, int64_t max_n, int max_r, int num_sms) {
  auto up = [](int64_t b) { return (b + 255) / 256 * 256; };
  const int64_t common = up(sizeof(PsgdState)) + up(sizeof(float) * 16 * 16) +
                         up(sizeof(uint32_t) * ceil_div(max_n, kStrip)) +
                         up(sizeof(uint32_t) * ceil_div(max_m, 8)) +
                         up(sizeof(float) * max_m * max_r) +
                         up(sizeof(double) * gram_parts_cap(max_m, num_sms) * max_r * max_r);
  // CUDA-core path: partial rows of P per column range, then the q
  // partials (splits * n * r floats with splits * strips <= 4 * SMs + strips)
  const int64_t cuda_core = up(sizeof(float) * kMaxColSplits * max_m * max_r) +
                            (int64_t)sizeof(float) * ((int64_t)num_sms * 4 * kStrip + max_n + kStrip) * max_r;
  // tensor-core path: one 128-row partial per (CTA, tile) pair, the images
  const int64_t tensor_core = tc_area_bytes(max_m, max_n, max_r, num_sms);
  return common + std::max(cuda_core, tensor_core);
}

gc_status launch_powersgd(gc_ctx* ctx, const float* grad, float* err, int64_t m,
                          int64_t n, int r, float* P_out, float* Q_inout) {
  if (m == 0 || n == 0) return GC_OK;
  switch (r) {
#define GC_R(RR) case RR: return run_psgd_r<RR>(ctx, grad, err, m, n, P_out, Q_inout);
    GC_R(1) GC_R(2) GC_R(3) GC_R(4) GC_R(5) GC_R(6) GC_R(7) GC_R(8)
    GC_R(9) GC_R(10) GC_R(11) GC_R(12) GC_R(13) GC_R(14) GC_R(15) GC_R(16)
#undef GC_R
    default: return GC_ERR_UNSUPPORTED;
  }
}

}  // namespace gc
