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
// the tensor-core ridge point, so the products run as fp32 FMAs on the CUDA
// cores and the kernels are organised around HBM streaming:
//   pass 1  mq       : M = G + E written over E; P = M Q (Q staged in shared
//                      memory).  Blocks own 16 rows and a range of columns
//                      (enough blocks to fill the GPU); the last block of a
//                      row range adds the column ranges' partial rows of P in
//                      order and forms their Gram matrix in fp64.  The last
//                      row range sums the Gram partials in order, factors
//                      P^T P = U^T U (Cholesky, fp64) and stores W = U^-1.
//                      P W is the Gram-Schmidt orthonormalisation of P: both
//                      give the unique QR factor with a positive diagonal.
//   pass 2  mtp      : Q' = M^T P_hat.  Blocks own a 128-column strip and a
//                      slice of rows; P_hat = P W for the slice is formed in
//                      shared memory (strip 0 also writes it out).  Partial
//                      sums are reduced in a fixed order by the last block of
//                      each strip, so results are deterministic.
//   pass 3  residual : E' = M - P_hat Q'^T (Q' staged in shared memory),
//                      blocks over rows and column ranges as in pass 1.
// Traffic: 12 + 4 + 8 = 24 bytes per element.
#include <algorithm>

#include "gc_internal.cuh"

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
  if (threadIdx.x == 0) {
    // Cholesky P^T P = U^T U (U upper, positive diagonal).  A column whose
    // remaining norm is 0 is dropped (its P_hat column is left zero), as
    // Gram-Schmidt leaves a zero column zero.
    double U[R][R], W[R][R];
    bool zero[R];
    for (int i = 0; i < R; ++i)
      for (int j = 0; j < R; ++j) U[i][j] = W[i][j] = 0.0;
    for (int j = 0; j < R; ++j) {
      for (int i = 0; i < j; ++i) {
        if (zero[i]) { U[i][j] = 0.0; continue; }
        double s = gram[i * R + j];
        for (int k = 0; k < i; ++k) s -= U[k][i] * U[k][j];
        U[i][j] = s / U[i][i];
      }
      double d = gram[j * R + j];
      for (int k = 0; k < j; ++k) d -= U[k][j] * U[k][j];
      zero[j] = !(d > 0.0);
      U[j][j] = zero[j] ? 1.0 : sqrt(d);
    }
    // W = U^-1 by back substitution, columns of dropped directions zero
    for (int j = R - 1; j >= 0; --j) {
      if (zero[j]) continue;
      W[j][j] = 1.0 / U[j][j];
      for (int i = j - 1; i >= 0; --i) {
        if (zero[i]) continue;
        double s = 0.0;
        for (int k = i + 1; k <= j; ++k) s += U[i][k] * W[k][j];
        W[i][j] = -s / U[i][i];
      }
    }
    for (int i = 0; i < R; ++i)
      for (int j = 0; j < R; ++j) b.w[i * R + j] = (float)W[i][j];
    b.state->ticket_mq = 0u;
  }
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
  b.state = static_cast<PsgdState*>(take(sizeof(PsgdState)));
  b.w = static_cast<float*>(take(sizeof(float) * 16 * 16));
  b.tickets = static_cast<uint32_t*>(take(sizeof(uint32_t) * ceil_div(pw.max_n, kStrip)));
  b.praw = static_cast<float*>(take(sizeof(float) * pw.max_m * pw.max_r));
  b.ppart = static_cast<float*>(take(sizeof(float) * kMaxColSplits * pw.max_m * pw.max_r));
  b.rb_tickets = static_cast<uint32_t*>(take(sizeof(uint32_t) * ceil_div(pw.max_m, kRowsPerBlock)));
  b.gram_part = static_cast<double*>(take(sizeof(double) * ceil_div(pw.max_m, kRowsPerBlock) * pw.max_r * pw.max_r));
  b.q_part = reinterpret_cast<float*>(base + off);
  b.status = ctx->ws.status;
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
  int64_t bytes = up(sizeof(PsgdState)) + up(sizeof(float) * 16 * 16) +
                  up(sizeof(uint32_t) * ceil_div(max_n, kStrip)) +
                  up(sizeof(float) * max_m * max_r) +
                  up(sizeof(float) * kMaxColSplits * max_m * max_r) +
                  up(sizeof(uint32_t) * ceil_div(max_m, kRowsPerBlock)) +
                  up(sizeof(double) * ceil_div(max_m, kRowsPerBlock) * max_r * max_r);
  // q partials: splits * n * r floats with splits * strips <= 4 * SMs + strips
  bytes += (int64_t)sizeof(float) * ((int64_t)num_sms * 4 * kStrip + max_n + kStrip) * max_r;
  return bytes;
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
