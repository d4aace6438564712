// Read accounting of the last decode and the kept-id gather used by the ABI.
#include "device_util.cuh"
#include "internal.cuh"

namespace mr {
namespace {

// ---------------------------------------------------------------------------
// Read accounting of the last decode (union over the batch).
// ---------------------------------------------------------------------------
__global__ void stats_mark_kernel(Dims d, int B, const int32_t* __restrict__ ids,
                                  const uint32_t* __restrict__ mask,
                                  const uint32_t* __restrict__ keptbits,
                                  uint32_t* __restrict__ bm_codes, uint32_t* __restrict__ bm_kept,
                                  uint32_t* __restrict__ bm_skip, uint32_t* __restrict__ bm_expert) {
  const int ts = blockIdx.x;   // t * topk + slot
  const int t = ts / d.topk, slot = ts % d.topk;
  const int e = ids[ts];
  if (threadIdx.x == 0) atomicOr(&bm_expert[e >> 5], 1u << (e & 31));
  for (int q = threadIdx.x; q < d.nb * 4; q += blockDim.x)
    atomicOr(&bm_codes[(size_t)e * d.nb * 4 + q], mask[(size_t)t * d.nb * 4 + q]);
  for (int wd = threadIdx.x; wd < d.I / 32; wd += blockDim.x) {
    const uint32_t kb = keptbits[(size_t)t * (d.N / 32) + slot * (d.I / 32) + wd];
    atomicOr(&bm_kept[(size_t)e * (d.I / 32) + wd], kb);
    atomicOr(&bm_skip[(size_t)e * (d.I / 32) + wd], ~kb);
  }
}

__global__ void stats_count_kernel(Dims d, const uint32_t* __restrict__ bm_codes,
                                   const uint32_t* __restrict__ bm_kept,
                                   const uint32_t* __restrict__ bm_skip,
                                   const uint32_t* __restrict__ bm_expert,
                                   unsigned long long* __restrict__ out) {
  // out: [0] coordinate runs, [1] kept rows, [2] skipped rows, [3] routed experts,
  //      [4] b sectors
  const long long gtid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  unsigned long long runs = 0, kr = 0, sr = 0, ex = 0, bsec = 0;
  for (long long q = gtid; q < (long long)d.E * d.nb * 4; q += nthreads) runs += __popc(bm_codes[q]);
  for (long long q = gtid; q < (long long)d.E * (d.I / 32); q += nthreads) {
    kr += __popc(bm_kept[q]);
    sr += __popc(bm_skip[q]);
  }
  for (long long q = gtid; q < (d.E + 31) / 32; q += nthreads) ex += __popc(bm_expert[q]);
  // b sectors: sector s of the b array covers bytes [32 s, 32 s + 32)
  const long long rowb = 2LL * d.r;
  const long long nsec = ((long long)d.E * d.I * rowb + 31) / 32;
  for (long long s = gtid; s < nsec; s += nthreads) {
    const long long r0 = (32 * s) / rowb, r1 = (32 * s + 31) / rowb;
    bool any = false;
    for (long long rr = r0; rr <= r1 && rr < (long long)d.E * d.I; ++rr)
      any |= (bm_skip[rr >> 5] >> (rr & 31)) & 1u;
    bsec += any;
  }
  if (runs) atomicAdd(&out[0], runs);
  if (kr) atomicAdd(&out[1], kr);
  if (sr) atomicAdd(&out[2], sr);
  if (ex) atomicAdd(&out[3], ex);
  if (bsec) atomicAdd(&out[4], bsec);
}

__global__ void gather_kept_kernel(Dims d, int B, int k, const int32_t* __restrict__ ids,
                                   const int32_t* __restrict__ kept, int32_t* __restrict__ out) {
  const long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= (long long)B * k) return;
  const int t = (int)(q / k), qi = (int)(q % k);
  const int n = kept[(size_t)t * d.N + qi];
  const int slot = n / d.I, i = n % d.I;
  out[q] = ids[t * d.topk + slot] * d.I + i;
}

}  // namespace

cudaError_t launch_stats(const moe_reader& h, int B, int k, cudaStream_t s) {
  const Dims& d = h.d;
  const Workspace& ws = h.ws;
  cudaError_t err;
  (void)k;
  if ((err = cudaMemsetAsync(ws.bm_codes, 0, (size_t)d.E * d.nb * 4 * 4, s)) != cudaSuccess) return err;
  if ((err = cudaMemsetAsync(ws.bm_kept, 0, (size_t)d.E * (d.I / 32) * 4, s)) != cudaSuccess) return err;
  if ((err = cudaMemsetAsync(ws.bm_skip, 0, (size_t)d.E * (d.I / 32) * 4, s)) != cudaSuccess) return err;
  if ((err = cudaMemsetAsync(ws.bm_expert, 0, (size_t)((d.E + 31) / 32) * 4, s)) != cudaSuccess) return err;
  if ((err = cudaMemsetAsync(ws.counters, 0, 16 * sizeof(unsigned long long), s)) != cudaSuccess) return err;
  if (B > 0) {
    stats_mark_kernel<<<B * d.topk, 128, 0, s>>>(d, B, ws.ids, ws.mask, ws.keptbits, ws.bm_codes,
                                                 ws.bm_kept, ws.bm_skip, ws.bm_expert);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    stats_count_kernel<<<152, 256, 0, s>>>(d, ws.bm_codes, ws.bm_kept, ws.bm_skip, ws.bm_expert,
                                           ws.counters);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  return cudaSuccess;
}

cudaError_t launch_gather_kept(const moe_reader& h, int B, int k, int32_t* out_dev, cudaStream_t s) {
  const long long n = (long long)B * k;
  if (n == 0) return cudaSuccess;
  gather_kept_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(h.d, B, k, h.ws.ids, h.ws.kept,
                                                                out_dev);
  return cudaGetLastError();
}

}  // namespace mr
