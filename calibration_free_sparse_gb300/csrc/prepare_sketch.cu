// Load-time kernels: rotated ternary sketch, down transpose, down norms and
// the recovery coefficients b_j.
//
// "Channel Selection for Mixture-of-Experts Decoding Needs No Calibration
// Data" (Chinese summary page, 方法步骤详情, load-time steps (1), (2), (4);
// 前置知识 "Hadamard旋转与三元Sketch" and "低秩恢复").
#include "device_util.cuh"
#include "internal.cuh"

namespace mr {
namespace {

// ---------------------------------------------------------------------------
// Rotate + ternarise + pack.
//
// One CTA = (expert e, block b, gate/up gv, chunk of 64 channels); 8 warps,
// each warp handles 8 consecutive channels (rows) one after another.  A row's
// 128-coordinate block lives in one warp: lane l holds coordinates
// l, l+32, l+64, l+96.  The Sylvester butterfly runs in fp64 (the BF16
// inputs make every butterfly sum exact), then w~ = z / sqrt(128) and the
// Ternary-Weight-Networks rule: Delta = 0.7 mean|w~|, t = sign(w~)[|w~| >
// Delta], alpha = mean of |w~| on the support (FP16), rho = mean (w~ -
// alpha t)^2 (FP16).  Codes of the 64 channels are staged per coordinate in
// shared memory and written as one 16-byte segment of each coordinate run.
// ---------------------------------------------------------------------------
constexpr int kSketchRowsPerWarp = 8;
constexpr int kSketchChunk = 64;

__global__ void __launch_bounds__(256)
sketch_kernel(Dims d, const __nv_bfloat16* __restrict__ G, const __nv_bfloat16* __restrict__ V,
              const int8_t* __restrict__ sigma, uint8_t* __restrict__ codes,
              __half* __restrict__ scales, __half* __restrict__ rho) {
  __shared__ __align__(16) uint8_t seg[kBlock][16];

  const int chunks = d.I / kSketchChunk;
  int idx = blockIdx.x;
  const int chunk = idx % chunks;
  idx /= chunks;
  const int gv = idx % 2;
  idx /= 2;
  const int b = idx % d.nb;
  const int e = idx / d.nb;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const __nv_bfloat16* W = gv ? V : G;

  double sg[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) sg[s] = (double)sigma[b * kBlock + lane + 32 * s];

  uint32_t packed[4] = {0u, 0u, 0u, 0u};   // bits 2r..2r+1 = code of row r (8 rows)
  const double sqrt128 = __dsqrt_rn(128.0);

  for (int r = 0; r < kSketchRowsPerWarp; ++r) {
    const int i = chunk * kSketchChunk + warp * kSketchRowsPerWarp + r;
    const __nv_bfloat16* row = W + ((size_t)e * d.I + i) * d.H;
    double u[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int col = b * kBlock + lane + 32 * s;
      const double v = col < d.H ? (double)__bfloat162float(row[col]) : 0.0;
      u[s] = sg[s] * v;
    }
    // butterflies over strides 1..16 (across lanes), then 32 and 64 (in lane)
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const double o = __shfl_xor_sync(0xffffffffu, u[s], h);
        u[s] = (lane & h) ? (o - u[s]) : (u[s] + o);
      }
    }
    {
      double a0 = u[0], a1 = u[1], a2 = u[2], a3 = u[3];
      u[0] = a0 + a1; u[1] = a0 - a1; u[2] = a2 + a3; u[3] = a2 - a3;
      a0 = u[0]; a1 = u[1]; a2 = u[2]; a3 = u[3];
      u[0] = a0 + a2; u[2] = a0 - a2; u[1] = a1 + a3; u[3] = a1 - a3;
    }
    double wt[4], aw[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      wt[s] = u[s] / sqrt128;
      aw[s] = fabs(wt[s]);
    }
    const double sumabs = warp_sum_d(aw[0] + aw[1] + aw[2] + aw[3]);
    const double delta = 0.7 * (sumabs / 128.0);
    int t[4];
    int nnz = 0;
    double sup = 0.0;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      t[s] = aw[s] > delta ? (wt[s] > 0.0 ? 1 : -1) : 0;
      nnz += t[s] != 0;
      sup += t[s] != 0 ? aw[s] : 0.0;
    }
    nnz = warp_sum_i(nnz);
    sup = warp_sum_d(sup);
    const double alpha = nnz > 0 ? sup / (double)nnz : 0.0;
    const __half a16 = f64_to_f16_rn(alpha);
    const double a16d = (double)__half2float(a16);
    double sq = 0.0;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const double res = wt[s] - a16d * (double)t[s];
      sq += res * res;
    }
    sq = warp_sum_d(sq);
    if (lane == 0) {
      const size_t o = (((size_t)e * d.nb + b) * 2 + gv) * d.I + i;
      scales[o] = a16;
      rho[o] = f64_to_f16_rn(sq / 128.0);
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const uint32_t q = t[s] == 0 ? 0u : (t[s] > 0 ? 1u : 3u);
      packed[s] |= q << (2 * r);
    }
  }
  // lane's coordinates c = lane + 32 s: bytes (2 warp, 2 warp + 1) of the segment
#pragma unroll
  for (int s = 0; s < 4; ++s)
    *reinterpret_cast<uint16_t*>(&seg[lane + 32 * s][2 * warp]) = (uint16_t)packed[s];
  __syncthreads();
  if (threadIdx.x < kBlock) {
    const int c = threadIdx.x;
    uint8_t* dst = codes + ((((size_t)e * d.nb + b) * kBlock + c) * 2 + gv) * d.S + chunk * 16;
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(&seg[c][0]);
  }
}

// ---------------------------------------------------------------------------
// D_e [H][I] -> Dt_e [I][H] through a 64x64 shared-memory tile.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
transpose_kernel(Dims d, const uint16_t* __restrict__ D, uint16_t* __restrict__ Dt) {
  __shared__ uint16_t tile[64][66];
  const int i0 = blockIdx.x * 64;
  const int h0 = blockIdx.y * 64;
  const int e = blockIdx.z;
  const uint16_t* src = D + (size_t)e * d.H * d.I;
  uint16_t* dst = Dt + (size_t)e * d.I * d.H;
  for (int q = threadIdx.x; q < 64 * 64; q += blockDim.x) {
    const int hh = q / 64, ii = q % 64;
    const int h = h0 + hh;
    tile[hh][ii] = h < d.H ? src[(size_t)h * d.I + i0 + ii] : (uint16_t)0;
  }
  __syncthreads();
  for (int q = threadIdx.x; q < 64 * 64; q += blockDim.x) {
    const int ii = q / 64, hh = q % 64;
    const int h = h0 + hh;
    if (h < d.H) dst[(size_t)(i0 + ii) * d.H + h] = tile[hh][ii];
  }
}

// ||d_j|| per channel: fp64 sum of squares of the BF16 column, stored fp32.
__global__ void __launch_bounds__(256)
dnorm_kernel(Dims d, const __nv_bfloat16* __restrict__ Dt, float* __restrict__ dnorm) {
  const int row = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= d.E * d.I) return;
  const __nv_bfloat16* p = Dt + (size_t)row * d.H;
  double acc = 0.0;
  for (int h = lane; h < d.H; h += 32) {
    const double v = (double)__bfloat162float(p[h]);
    acc += v * v;
  }
  acc = warp_sum_d(acc);
  if (lane == 0) dnorm[row] = __double2float_rn(__dsqrt_rn(acc));
}

// ||b_j||^2 of the stored FP16 coefficients, one thread per channel.
__global__ void bnorm2_kernel(Dims d, const __half* __restrict__ b, float* __restrict__ out) {
  const long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= (long long)d.E * d.I) return;
  float s = 0.f;
  for (int j = 0; j < d.r; ++j) {
    const float v = __half2float(b[q * d.r + j]);
    s = fmaf(v, v, s);
  }
  out[q] = s;
}

// b_j = U^T d_j for every channel (FP16 U, BF16 d, fp32 accumulation of
// exact products, FP16 result).  CTA = 64 channels; tiles of 128 coordinates.
constexpr int kBRows = 64;
constexpr int kBTile = 128;

__global__ void __launch_bounds__(256)
project_b_kernel(Dims d, const __nv_bfloat16* __restrict__ Dt, const __half* __restrict__ U,
                 __half* __restrict__ bout) {
  __shared__ float Ds[kBRows][kBTile + 1];
  __shared__ float Us[kBTile][kMaxRank];
  const int q0 = blockIdx.x * kBRows;
  const int t = threadIdx.x;
  const int row = t >> 2;          // 0..63
  const int jg = t & 3;            // j = jg + 4 m
  float acc[kMaxRank / 4];
#pragma unroll
  for (int m = 0; m < kMaxRank / 4; ++m) acc[m] = 0.f;
  const int total = d.E * d.I;

  for (int h0 = 0; h0 < d.H; h0 += kBTile) {
    for (int q = t; q < kBRows * kBTile; q += blockDim.x) {
      const int rr = q / kBTile, hh = q % kBTile;
      const int qq = q0 + rr, h = h0 + hh;
      Ds[rr][hh] = (qq < total && h < d.H) ? __bfloat162float(Dt[(size_t)qq * d.H + h]) : 0.f;
    }
    for (int q = t; q < kBTile * d.r; q += blockDim.x) {
      const int hh = q / d.r, j = q % d.r;
      const int h = h0 + hh;
      Us[hh][j] = h < d.H ? __half2float(U[(size_t)h * d.r + j]) : 0.f;
    }
    __syncthreads();
    for (int hh = 0; hh < kBTile; ++hh) {
      const float dv = Ds[row][hh];
#pragma unroll
      for (int m = 0; m < kMaxRank / 4; ++m) {
        const int j = jg + 4 * m;
        if (j < d.r) acc[m] = fmaf(dv, Us[hh][j], acc[m]);
      }
    }
    __syncthreads();
  }
  const int qq = q0 + row;
  if (qq < total) {
#pragma unroll
    for (int m = 0; m < kMaxRank / 4; ++m) {
      const int j = jg + 4 * m;
      if (j < d.r) bout[(size_t)qq * d.r + j] = __float2half_rn(acc[m]);
    }
  }
}

// ---------------------------------------------------------------------------
// Five trits per byte: output byte j of a run holds channels 5j .. 5j+4 as
// sum_m digit * 3^m (2-bit code 0b00 -> 0, 0b01 (+1) -> 1, 0b11 (-1) -> 2);
// channels past I and the sector padding are 0.  A thread per output byte.
// ---------------------------------------------------------------------------
__global__ void pack_trit5_kernel(Dims d, const uint8_t* __restrict__ codes2,
                                  uint8_t* __restrict__ codes5, long long runs) {
  const long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= runs * d.S) return;
  const long long run = q / d.S;
  const int j = (int)(q - run * d.S);
  const uint8_t* src = codes2 + run * d.S2b;
  int v = 0, p3 = 1;
#pragma unroll
  for (int m = 0; m < 5; ++m) {
    const int i = 5 * j + m;
    if (i < d.I) {
      const int c = (src[i >> 2] >> (2 * (i & 3))) & 3;
      v += (c == 1 ? 1 : (c == 3 ? 2 : 0)) * p3;
    }
    p3 *= 3;
  }
  codes5[q] = (uint8_t)v;
}

}  // namespace

cudaError_t launch_pack_trit5(const Dims& d, const uint8_t* codes2, uint8_t* codes5, cudaStream_t s) {
  const long long runs = (long long)d.E * d.nb * kBlock * 2;
  const long long n = runs * d.S;
  pack_trit5_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(d, codes2, codes5, runs);
  return cudaGetLastError();
}

// Ut[j][h] = U[h][j]: the output phase reads rank components as rows.
__global__ void transpose_u_kernel(int H, int r, const __half* __restrict__ U,
                                   __half* __restrict__ Ut) {
  const int q = blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= H * r) return;
  const int j = q / H, h = q % H;
  Ut[q] = U[(size_t)h * r + j];
}

cudaError_t launch_sketch(const Dims& d, const __nv_bfloat16* G, const __nv_bfloat16* V,
                          const int8_t* sigma, uint8_t* codes, __half* scales, __half* rho,
                          cudaStream_t s) {
  const size_t code_bytes = (size_t)d.E * d.nb * kBlock * 2 * d.S;
  cudaError_t err = cudaMemsetAsync(codes, 0, code_bytes, s);
  if (err != cudaSuccess) return err;
  const long long grid = (long long)d.E * d.nb * 2 * (d.I / kSketchChunk);
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  sketch_kernel<<<(unsigned)grid, 256, 0, s>>>(d, G, V, sigma, codes, scales, rho);
  return cudaGetLastError();
}

cudaError_t launch_transpose_down(const Dims& d, const __nv_bfloat16* D, __nv_bfloat16* Dt,
                                  cudaStream_t s) {
  dim3 grid(d.I / 64, (d.H + 63) / 64, d.E);
  transpose_kernel<<<grid, 256, 0, s>>>(d, reinterpret_cast<const uint16_t*>(D),
                                        reinterpret_cast<uint16_t*>(Dt));
  return cudaGetLastError();
}

cudaError_t launch_dnorm(const Dims& d, const __nv_bfloat16* Dt, float* dnorm, cudaStream_t s) {
  const int rows = d.E * d.I;
  dnorm_kernel<<<(rows + 7) / 8, 256, 0, s>>>(d, Dt, dnorm);
  return cudaGetLastError();
}

cudaError_t launch_transpose_u(const Dims& d, const __half* U, __half* Ut, cudaStream_t s) {
  const int n = d.H * d.r;
  transpose_u_kernel<<<(n + 255) / 256, 256, 0, s>>>(d.H, d.r, U, Ut);
  return cudaGetLastError();
}

cudaError_t launch_bnorm2(const Dims& d, const __half* b, float* bnorm2, cudaStream_t s) {
  const long long n = (long long)d.E * d.I;
  bnorm2_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(d, b, bnorm2);
  return cudaGetLastError();
}

cudaError_t launch_project_b(const Dims& d, const __nv_bfloat16* Dt, const __half* U, __half* b,
                             cudaStream_t s) {
  const int rows = d.E * d.I;
  project_b_kernel<<<(rows + kBRows - 1) / kBRows, 256, 0, s>>>(d, Dt, U, b);
  return cudaGetLastError();
}

}  // namespace mr
