// Load-time recovery basis: U = top-r left singular vectors of the layer's
// stacked down columns ("Channel Selection for Mixture-of-Experts Decoding
// Needs No Calibration Data", Chinese summary page, 前置知识 "低秩恢复" and
// 方法步骤详情 load-time step (3)).
//
// They are the top-r eigenvectors of M = sum_j d_j d_j^T (H x H):
//   1. gram_kernel        M from Dt (exact BF16 products, fp32 tile sums,
//                         fp64 accumulation across tiles)
//   2. tridiag_kernel     fp64 Householder reduction M = Q T Q^T in one
//                         cooperative kernel (two bounded grid barriers/step)
//   3. bisect_kernel      top-r eigenvalues of T by Sturm-count bisection
//   4. inverse_iter_kernel eigenvectors of T by inverse iteration (LU with
//                         partial pivoting of the tridiagonal)
//   5. mgs_kernel         re-orthonormalise the r vectors
//   6. backtransform_kernel  apply Q
//   7. canonical_kernel   sign (largest-|.| entry positive) and FP16 rounding
#include <float.h>

#include "device_util.cuh"
#include "internal.cuh"

namespace mr {
namespace {

// ---------------------------------------------------------------------------
// Gram: M[h1][h2] += sum_q Dt[q][h1] Dt[q][h2] over a K-chunk of channels.
// 64x64 output tile per CTA (lower-triangular tile pairs only), 4x4 per thread.
// ---------------------------------------------------------------------------
constexpr int kGT = 64;
constexpr int kGK = 32;
constexpr int kGChunk = 1024;

__global__ void __launch_bounds__(256)
gram_kernel(int H, int K, const __nv_bfloat16* __restrict__ Dt, double* __restrict__ M) {
  __shared__ float As[kGK][kGT];
  __shared__ float Bs[kGK][kGT];
  // tile pair (ti >= tj) from the linear index
  int lin = blockIdx.x;
  int ti = 0;
  while (lin > ti) { lin -= ti + 1; ++ti; }
  const int tj = lin;
  const int k0 = blockIdx.y * kGChunk;
  const int k1 = min(K, k0 + kGChunk);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;

  for (int kk = k0; kk < k1; kk += kGK) {
    for (int q = threadIdx.x; q < kGK * kGT; q += blockDim.x) {
      const int r = q / kGT, c = q % kGT;
      const int krow = kk + r;
      const int ha = ti * kGT + c, hb = tj * kGT + c;
      const bool okr = krow < k1;
      As[r][c] = (okr && ha < H) ? __bfloat162float(Dt[(size_t)krow * H + ha]) : 0.f;
      Bs[r][c] = (okr && hb < H) ? __bfloat162float(Dt[(size_t)krow * H + hb]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int r = 0; r < kGK; ++r) {
      float av[4], bv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) av[a] = As[r][ty * 4 + a];
#pragma unroll
      for (int b = 0; b < 4; ++b) bv[b] = Bs[r][tx * 4 + b];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(av[a], bv[b], acc[a][b]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int h1 = ti * kGT + ty * 4 + a, h2 = tj * kGT + tx * 4 + b;
      if (h1 < H && h2 < H) {
        atomicAdd(&M[(size_t)h1 * H + h2], (double)acc[a][b]);
        if (ti != tj) atomicAdd(&M[(size_t)h2 * H + h1], (double)acc[a][b]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Bounded grid barrier for a cooperative launch.  Every wait has an
// iteration limit; on timeout the abort flag is raised and all CTAs leave.
// ---------------------------------------------------------------------------
struct GridSync {
  unsigned int count;
  unsigned int gen;
  unsigned int abort;
  unsigned int pad;
};

constexpr unsigned long long kBarrierNs = 1000000000ull;   // one second of the global timer

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ bool grid_barrier(GridSync* gs, unsigned int nblocks) {
  __shared__ int ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile unsigned int* vgen = &gs->gen;
    volatile unsigned int* vab = &gs->abort;
    const unsigned int gen = *vgen;
    __threadfence();
    const unsigned int arrived = atomicAdd(&gs->count, 1u);
    if (arrived == nblocks - 1) {
      atomicExch(&gs->count, 0u);
      __threadfence();
      atomicAdd(&gs->gen, 1u);
    } else {
      const unsigned long long t0 = global_ns();
      while (*vgen == gen) {
        if (*vab) break;
        if (global_ns() - t0 > kBarrierNs) {
          atomicExch(&gs->abort, 1u);
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
    ok = *vab == 0u;
  }
  __syncthreads();
  return ok != 0;
}

__device__ double block_sum_d(double v, double* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum_d(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  double s = 0.0;
  for (int i = 0; i < nw; ++i) s += red[i];   // same order in every CTA
  __syncthreads();
  return s;
}

// ---------------------------------------------------------------------------
// Householder tridiagonalisation of the symmetric n x n matrix A (row-major,
// both triangles kept).  Step k: x = A[k][k+1:], beta = -sign(x0)||x||,
// tau = (beta - x0)/beta, v = [1, x[1:]/(x0 - beta)], p = tau A22 v,
// w = p - (tau/2)(p.v) v, A22 -= v w^T + w v^T.  Row k keeps x for the back
// transformation (tau_k, scale_k = 1/(x0 - beta) are stored).
// Rows are owned by warps across the grid (row i -> warp (i - k - 1) mod W).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(512)
tridiag_kernel(int n, double* __restrict__ A, double* __restrict__ dg, double* __restrict__ eg,
               double* __restrict__ tau, double* __restrict__ vscale, double* __restrict__ p,
               double* __restrict__ part, GridSync* gs, uint32_t* err, unsigned int extra) {
  extern __shared__ double sm[];
  double* v = sm;            // [n]
  double* w = sm + n;        // [n]
  double* red = sm + 2 * n;  // [32]
  __shared__ double bcast;
  const unsigned int P = gridDim.x;
  const unsigned int arrivals = P + extra;   // extra > 0 only under fault injection
  const int warps = blockDim.x >> 5, wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Wtot = (int)P * warps;
  const int gw = blockIdx.x * warps + wid;

  for (int k = 0; k + 2 < n; ++k) {
    const double* rowk = A + (size_t)k * n;
    double s = 0.0;
    for (int j = k + 2 + threadIdx.x; j < n; j += blockDim.x) {
      const double t = __ldcg(rowk + j);
      s += t * t;
    }
    s = block_sum_d(s, red);
    const double alpha = __ldcg(rowk + k + 1);
    double beta, tk, scale;
    if (s == 0.0) {
      tk = 0.0;
      beta = alpha;
      scale = 0.0;
    } else {
      beta = -copysign(sqrt(alpha * alpha + s), alpha);
      tk = (beta - alpha) / beta;
      scale = 1.0 / (alpha - beta);
    }
    for (int j = k + 1 + threadIdx.x; j < n; j += blockDim.x)
      v[j - k - 1] = (j == k + 1) ? 1.0 : __ldcg(rowk + j) * scale;
    __syncthreads();

    double pv = 0.0;
    for (int i = k + 1 + gw; i < n; i += Wtot) {
      const double* rowi = A + (size_t)i * n;
      double acc = 0.0;
      for (int j = k + 1 + lane; j < n; j += 32) acc += __ldcg(rowi + j) * v[j - k - 1];
      acc = warp_sum_d(acc) * tk;
      if (lane == 0) __stcg(p + i, acc);
      pv += acc * v[i - k - 1];
    }
    if (lane == 0) red[wid] = pv;
    __syncthreads();
    if (threadIdx.x == 0) {
      double t = 0.0;
      for (int q = 0; q < warps; ++q) t += red[q];
      __stcg(part + blockIdx.x, t);
    }
    if (!grid_barrier(gs, arrivals)) goto fail;

    if (threadIdx.x == 0) {
      double t = 0.0;
      for (unsigned int q = 0; q < P; ++q) t += __ldcg(part + q);
      bcast = 0.5 * tk * t;
    }
    __syncthreads();
    {
      const double K = bcast;
      for (int j = k + 1 + threadIdx.x; j < n; j += blockDim.x)
        w[j - k - 1] = __ldcg(p + j) - K * v[j - k - 1];
    }
    __syncthreads();
    for (int i = k + 1 + gw; i < n; i += Wtot) {
      double* rowi = A + (size_t)i * n;
      const double vi = v[i - k - 1], wi = w[i - k - 1];
      for (int j = k + 1 + lane; j < n; j += 32) {
        const double a = __ldcg(rowi + j) - (vi * w[j - k - 1] + wi * v[j - k - 1]);
        __stcg(rowi + j, a);
      }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      dg[k] = __ldcg(A + (size_t)k * n + k);
      eg[k] = beta;
      tau[k] = tk;
      vscale[k] = scale;
    }
    if (!grid_barrier(gs, arrivals)) goto fail;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (n >= 2) {
      dg[n - 2] = __ldcg(A + (size_t)(n - 2) * n + (n - 2));
      eg[n - 2] = __ldcg(A + (size_t)(n - 2) * n + (n - 1));
      tau[n - 2] = 0.0;
      vscale[n - 2] = 0.0;
    }
    dg[n - 1] = __ldcg(A + (size_t)(n - 1) * n + (n - 1));
  }
  return;
fail:
  if (threadIdx.x == 0) atomicOr(err, kErrTimeout);
}

// Sturm count: number of eigenvalues of T strictly below x.
__device__ int sturm_count(int n, const double* dg, const double* e2, double x, double pivmin) {
  int cnt = 0;
  double q = dg[0] - x;
  if (fabs(q) < pivmin) q = -pivmin;
  cnt += q < 0.0;
  for (int i = 1; i < n; ++i) {
    q = (dg[i] - x) - e2[i - 1] / q;
    if (fabs(q) < pivmin) q = -pivmin;
    cnt += q < 0.0;
  }
  return cnt;
}

// e2[i] = eg[i]^2 (one thread per entry).
__global__ void square_offdiag_kernel(int n, const double* __restrict__ eg, double* __restrict__ e2) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i + 1 < n) e2[i] = eg[i] * eg[i];
}

// Warp j finds the j-th largest eigenvalue of T = tridiag(e, dg, e) by
// multisection: each step its 32 lanes take Sturm counts at 32 points that
// split [lo, hi] into 33 equal parts, and the part holding the eigenvalue
// becomes the new interval; it stops when the points no longer fall strictly
// inside the interval (the interval is down to a few ulps).
__global__ void bisect_kernel(int n, int r, const double* __restrict__ dg,
                              const double* __restrict__ eg, const double* __restrict__ e2,
                              double* __restrict__ lam) {
  const int j = blockIdx.x, lane = threadIdx.x;
  if (j >= r) return;
  double lo = DBL_MAX, hi = -DBL_MAX, emax2 = 0.0;
  for (int i = lane; i < n; i += 32) {
    const double a = i > 0 ? fabs(eg[i - 1]) : 0.0;
    const double b = i + 1 < n ? fabs(eg[i]) : 0.0;
    lo = fmin(lo, dg[i] - a - b);
    hi = fmax(hi, dg[i] + a + b);
    if (i + 1 < n) emax2 = fmax(emax2, e2[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = fmin(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = fmax(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    emax2 = fmax(emax2, __shfl_xor_sync(0xffffffffu, emax2, o));
  }
  const double span = fmax(hi - lo, fmax(fabs(lo), fabs(hi)) * DBL_EPSILON);
  lo -= 2.0 * DBL_EPSILON * span + DBL_MIN;
  hi += 2.0 * DBL_EPSILON * span + DBL_MIN;
  const double pivmin = DBL_MIN * fmax(1.0, emax2);
  const int target = n - 1 - j;   // eigenvalues strictly below the wanted one
  for (int it = 0; it < 64; ++it) {
    const double x = lo + (hi - lo) * ((double)(lane + 1) / 33.0);
    const bool inside = x > lo && x < hi;
    if (!__all_sync(0xffffffffu, inside)) break;
    const bool above = sturm_count(n, dg, e2, x, pivmin) >= target + 1;   // eigenvalue < x
    const unsigned bal = __ballot_sync(0xffffffffu, above);
    const int first = bal ? __ffs(bal) - 1 : 32;   // the first point above the eigenvalue
    const double xhi = __shfl_sync(0xffffffffu, x, first < 32 ? first : 31);
    const double xlo = __shfl_sync(0xffffffffu, x, first > 0 ? first - 1 : 0);
    if (first < 32) hi = xhi;
    if (first > 0) lo = xlo;
  }
  // finish by bisection while a midpoint still falls strictly inside
  for (int it = 0; it < 128; ++it) {
    const double mid = 0.5 * (lo + hi);
    if (mid <= lo || mid >= hi) break;
    if (sturm_count(n, dg, e2, mid, pivmin) >= target + 1)
      hi = mid;
    else
      lo = mid;
  }
  if (lane == 0) lam[j] = 0.5 * (lo + hi);
}

// Inverse iteration for eigenvalue lam[j] of T (thread j); scratch holds
// five length-n arrays per thread: a, dl, du, du2 and the iterate z.
__global__ void inverse_iter_kernel(int n, int r, const double* __restrict__ dg,
                                    const double* __restrict__ eg, const double* __restrict__ lam,
                                    double* __restrict__ scratch, unsigned char* __restrict__ piv,
                                    double* __restrict__ Z) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= r) return;
  double* a = scratch + (size_t)j * 4 * n;
  double* dl = a + n;
  double* du = dl + n;
  double* du2 = du + n;
  unsigned char* pv = piv + (size_t)j * n;
  double* z = Z + (size_t)j * n;
  const double x = lam[j];
  double tnorm = 0.0;
  for (int i = 0; i < n; ++i) {
    a[i] = dg[i] - x;
    if (i + 1 < n) {
      dl[i] = eg[i];
      du[i] = eg[i];
    }
    du2[i] = 0.0;
    tnorm = fmax(tnorm, fabs(dg[i]) + (i > 0 ? fabs(eg[i - 1]) : 0.0) + (i + 1 < n ? fabs(eg[i]) : 0.0));
  }
  const double tiny = DBL_EPSILON * fmax(tnorm, DBL_MIN);
  // LU with partial pivoting of the tridiagonal (row interchanges between i, i+1)
  for (int i = 0; i + 1 < n; ++i) {
    if (fabs(a[i]) >= fabs(dl[i])) {
      pv[i] = 0;
      if (a[i] != 0.0) {
        const double f = dl[i] / a[i];
        dl[i] = f;
        a[i + 1] -= f * du[i];
      } else {
        dl[i] = 0.0;
      }
      du2[i] = 0.0;
    } else {
      pv[i] = 1;
      const double f = a[i] / dl[i];
      a[i] = dl[i];
      dl[i] = f;
      const double t = du[i];
      du[i] = a[i + 1];
      a[i + 1] = t - f * a[i + 1];
      if (i + 2 < n) {
        du2[i] = du[i + 1];
        du[i + 1] = -f * du[i + 1];
      } else {
        du2[i] = 0.0;
      }
    }
  }
  for (int i = 0; i < n; ++i)
    if (fabs(a[i]) < tiny) a[i] = a[i] < 0.0 ? -tiny : tiny;
  // deterministic start vector in [-1, 1]
  for (int i = 0; i < n; ++i) {
    const unsigned int hsh = (unsigned int)(i + 1) * 2654435761u ^ (unsigned int)(j + 7) * 40503u;
    z[i] = (double)(hsh % 2001u) / 1000.0 - 1.0 + 1e-3;
  }
  for (int it = 0; it < 3; ++it) {
    for (int i = 0; i + 1 < n; ++i) {
      if (pv[i] == 0) {
        z[i + 1] -= dl[i] * z[i];
      } else {
        const double t = z[i];
        z[i] = z[i + 1];
        z[i + 1] = t - dl[i] * z[i];
      }
    }
    z[n - 1] /= a[n - 1];
    if (n >= 2) z[n - 2] = (z[n - 2] - du[n - 2] * z[n - 1]) / a[n - 2];
    for (int i = n - 3; i >= 0; --i) z[i] = (z[i] - du[i] * z[i + 1] - du2[i] * z[i + 2]) / a[i];
    double nrm = 0.0, zmax = 0.0;
    for (int i = 0; i < n; ++i) zmax = fmax(zmax, fabs(z[i]));
    if (zmax == 0.0) zmax = 1.0;
    for (int i = 0; i < n; ++i) {
      z[i] /= zmax;
      nrm += z[i] * z[i];
    }
    nrm = sqrt(nrm);
    for (int i = 0; i < n; ++i) z[i] /= nrm;
  }
}

// Modified Gram-Schmidt over the r eigenvectors of T (one CTA).
__global__ void __launch_bounds__(1024)
mgs_kernel(int n, int r, double* __restrict__ Z) {
  __shared__ double red[32];
  for (int j = 0; j < r; ++j) {
    double* zj = Z + (size_t)j * n;
    for (int i = 0; i < j; ++i) {
      const double* zi = Z + (size_t)i * n;
      double s = 0.0;
      for (int q = threadIdx.x; q < n; q += blockDim.x) s += zi[q] * zj[q];
      s = block_sum_d(s, red);
      for (int q = threadIdx.x; q < n; q += blockDim.x) zj[q] -= s * zi[q];
      __syncthreads();
    }
    double s = 0.0;
    for (int q = threadIdx.x; q < n; q += blockDim.x) s += zj[q] * zj[q];
    s = block_sum_d(s, red);
    const double inv = 1.0 / sqrt(s);
    for (int q = threadIdx.x; q < n; q += blockDim.x) zj[q] *= inv;
    __syncthreads();
  }
}

// Q z for one eigenvector per CTA: apply H_k = I - tau_k v_k v_k^T for
// k = n-3 .. 0, v_k = [1 at k+1, scale_k * A[k][k+2:]].
__global__ void __launch_bounds__(512)
backtransform_kernel(int n, const double* __restrict__ A, const double* __restrict__ tau,
                     const double* __restrict__ vscale, double* __restrict__ Z) {
  extern __shared__ double z[];
  __shared__ double red[32];
  double* zg = Z + (size_t)blockIdx.x * n;
  for (int q = threadIdx.x; q < n; q += blockDim.x) z[q] = zg[q];
  __syncthreads();
  for (int k = n - 3; k >= 0; --k) {
    const double tk = tau[k];
    if (tk == 0.0) continue;
    const double sc = vscale[k];
    const double* rowk = A + (size_t)k * n;
    const double zk1 = z[k + 1];
    double s = 0.0;
    for (int q = k + 2 + threadIdx.x; q < n; q += blockDim.x) s += sc * rowk[q] * z[q];
    s = block_sum_d(s, red);   // ends with a barrier: every thread has read zk1
    s = tk * (s + zk1);
    for (int q = k + 2 + threadIdx.x; q < n; q += blockDim.x) z[q] -= s * sc * rowk[q];
    if (threadIdx.x == 0) z[k + 1] = zk1 - s;
    __syncthreads();
  }
  for (int q = threadIdx.x; q < n; q += blockDim.x) zg[q] = z[q];
}

// Canonical sign (largest-magnitude entry positive, first index on ties)
// and FP16 rounding into U [H][r]; one warp per column.
__global__ void canonical_kernel(int n, int r, const double* __restrict__ Z, __half* __restrict__ U) {
  const int j = blockIdx.x;
  const int lane = threadIdx.x;
  const double* z = Z + (size_t)j * n;
  double best = -1.0;
  int bi = 0x7fffffff;
  for (int q = lane; q < n; q += 32) {
    const double a = fabs(z[q]);
    if (a > best) {
      best = a;
      bi = q;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ob > best || (ob == best && oi < bi)) {
      best = ob;
      bi = oi;
    }
  }
  const double sgn = z[bi] < 0.0 ? -1.0 : 1.0;
  for (int q = lane; q < n; q += 32) U[(size_t)q * r + j] = f64_to_f16_rn(sgn * z[q]);
}

}  // namespace

int build_recovery_basis(const Dims& d, const __nv_bfloat16* Dt, __half* U, double* eigvals,
                         cudaStream_t s, bool stall) {
  const int n = d.H, r = d.r, K = d.E * d.I;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_READER_ECUDA;
  int sms = 0, coop = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  if (!coop || sms <= 0) return MOE_READER_ECUDA;

  // scratch: M (n*n), dg, eg, tau, vscale, p (n each), part (sms), e2 (n), lam (r),
  // inverse-iteration arrays (4 n r), Z (n r), pivots (n r bytes), barrier, error word
  const size_t nn = (size_t)n * n;
  const size_t doubles = nn + 6 * (size_t)n + (size_t)sms + (size_t)r + 4 * (size_t)n * r +
                         (size_t)n * r;
  const size_t bytes = doubles * sizeof(double) + (size_t)n * r + sizeof(GridSync) + 64;
  void* base = nullptr;
  {
    const cudaError_t ae = device_alloc(&base, bytes);
    if (ae == cudaErrorMemoryAllocation) return MOE_READER_ENOMEM;
    if (ae != cudaSuccess) return MOE_READER_ECUDA;
  }
  double* M = static_cast<double*>(base);
  double* dg = M + nn;
  double* eg = dg + n;
  double* tau = eg + n;
  double* vsc = tau + n;
  double* p = vsc + n;
  double* e2 = p + n;
  double* part = e2 + n;
  double* lam = part + sms;
  double* scr = lam + r;
  double* Z = scr + 4 * (size_t)n * r;
  unsigned char* piv = reinterpret_cast<unsigned char*>(Z + (size_t)n * r);
  uintptr_t gsp = reinterpret_cast<uintptr_t>(piv + (size_t)n * r);
  gsp = (gsp + 15) & ~(uintptr_t)15;
  GridSync* gs = reinterpret_cast<GridSync*>(gsp);
  uint32_t* err = reinterpret_cast<uint32_t*>(gs + 1);

  int status = MOE_READER_OK;
  cudaError_t ce = cudaSuccess;
  do {
    if ((ce = cudaMemsetAsync(base, 0, bytes, s)) != cudaSuccess) break;
    const int tiles = (n + kGT - 1) / kGT;
    dim3 ggrid(tiles * (tiles + 1) / 2, (K + kGChunk - 1) / kGChunk);
    gram_kernel<<<ggrid, 256, 0, s>>>(n, K, Dt, M);
    if ((ce = cudaGetLastError()) != cudaSuccess) break;

    const size_t smem = (2 * (size_t)n + 32) * sizeof(double);
    if ((ce = cudaFuncSetAttribute(tridiag_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)smem)) != cudaSuccess)
      break;
    int per_sm = 0;
    if ((ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tridiag_kernel, 512, smem)) !=
        cudaSuccess)
      break;
    if (per_sm < 1) {
      ce = cudaErrorInvalidConfiguration;
      break;
    }
    const int grid = sms;   // one CTA per SM: co-resident under a cooperative launch
    int nn_arg = n;
    unsigned int extra = stall ? 1u : 0u;
    void* args[] = {&nn_arg, &M, &dg, &eg, &tau, &vsc, &p, &part, &gs, &err, &extra};
    if ((ce = cudaLaunchCooperativeKernel((void*)tridiag_kernel, dim3(grid), dim3(512), args, smem,
                                          s)) != cudaSuccess)
      break;
    square_offdiag_kernel<<<(n + 255) / 256, 256, 0, s>>>(n, eg, e2);
    if ((ce = cudaGetLastError()) != cudaSuccess) break;
    bisect_kernel<<<r, 32, 0, s>>>(n, r, dg, eg, e2, lam);
    if ((ce = cudaGetLastError()) != cudaSuccess) break;
    inverse_iter_kernel<<<(r + 31) / 32, 32, 0, s>>>(n, r, dg, eg, lam, scr, piv, Z);
    if ((ce = cudaGetLastError()) != cudaSuccess) break;
    mgs_kernel<<<1, 1024, 0, s>>>(n, r, Z);
    if ((ce = cudaGetLastError()) != cudaSuccess) break;
    const size_t bsm = (size_t)n * sizeof(double);
    if ((ce = cudaFuncSetAttribute(backtransform_kernel,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bsm)) !=
        cudaSuccess)
      break;
    backtransform_kernel<<<r, 512, bsm, s>>>(n, M, tau, vsc, Z);
    if ((ce = cudaGetLastError()) != cudaSuccess) break;
    canonical_kernel<<<r, 32, 0, s>>>(n, r, Z, U);
    if ((ce = cudaGetLastError()) != cudaSuccess) break;
    if ((ce = cudaMemcpyAsync(eigvals, lam, (size_t)r * sizeof(double), cudaMemcpyDeviceToDevice,
                              s)) != cudaSuccess)
      break;
    uint32_t herr = 0;
    if ((ce = cudaMemcpyAsync(&herr, err, sizeof(uint32_t), cudaMemcpyDeviceToHost, s)) !=
        cudaSuccess)
      break;
    if ((ce = cudaStreamSynchronize(s)) != cudaSuccess) break;
    if (herr & kErrTimeout) status = MOE_READER_ETIMEOUT;
  } while (0);
  if (ce != cudaSuccess) {
    status = MOE_READER_ECUDA;
    cudaStreamSynchronize(s);
  }
  cudaFree(base);
  return status;
}

}  // namespace mr
