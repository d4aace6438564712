// Exact per-row top-k selection that allocates nothing.
//
// This is the selection step of the decode (largest score first, lower id on
// ties) offered on its own for callers that cannot call cudaMalloc: code
// running inside CUDA-graph stream capture, inference-engine plugins that may
// only use memory the engine hands them, and hosts whose allocator forbids
// device allocations after start-up.  Its scratch lives in one file-scope
// __device__ array of fixed size instead of a handle's workspace.
#include <mutex>

#include "internal.cuh"

namespace {

// Scratch capacity in elements (rows x columns); 9 bytes per element: the
// order key, the tie key and a candidate flag.  About 2.3 MiB, held by every
// GPU that loads the library until the process exits.
constexpr long long kNoAllocMaxElems = 1LL << 18;
constexpr int kNoAllocMaxDevices = 64;

__device__ __align__(256) unsigned char g_topk_scratch[kNoAllocMaxElems * 9];

std::mutex g_setup_mu;
void* g_scratch_ptr[kNoAllocMaxDevices];
bool g_scratch_ready[kNoAllocMaxDevices];

// Order-preserving map of an fp32 value to uint32 (larger float -> larger
// key).  Values that compare equal get equal keys: -0 maps like +0, and every
// NaN (either sign, any payload) maps to the largest key, above +infinity.
__device__ __forceinline__ uint32_t order_key(float f) {
  if (f != f) return 0xffffffffu;
  const uint32_t u = __float_as_uint(f == 0.f ? 0.f : f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// k-th largest key among the valid entries of one row; *rem = how many entries
// equal to the returned key are needed to reach k.
__device__ uint32_t row_radix_select(const uint32_t* keys, const uint8_t* valid, int N, int kth,
                                     int* hist, int* sh, int* rem) {
  uint32_t prefix = 0, pmask = 0;
  int remaining = kth;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int n = threadIdx.x; n < N; n += blockDim.x) {
      if (valid && !__ldcg(valid + n)) continue;
      const uint32_t kk = __ldcg(keys + n);
      if ((kk & pmask) == prefix) atomicAdd(&hist[(kk >> shift) & 255u], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int above = 0, d = 255;
      for (; d > 0; --d) {
        if (above + hist[d] >= remaining) break;
        above += hist[d];
      }
      sh[0] = d;
      sh[1] = remaining - above;
    }
    __syncthreads();
    prefix |= (uint32_t)sh[0] << shift;
    pmask |= 255u << shift;
    remaining = sh[1];
    __syncthreads();
  }
  *rem = remaining;
  return prefix;
}

__global__ void __launch_bounds__(1024)
topk_noalloc_kernel(const float* __restrict__ scores, const int32_t* __restrict__ ids, int N,
                    int k, int32_t* __restrict__ kept, unsigned char* __restrict__ scratch,
                    long long total) {
  __shared__ int hist[256];
  __shared__ int sh[2];
  __shared__ int wsum[32];
  __shared__ int wsum2[32];
  const int row = blockIdx.x;
  uint32_t* keys = reinterpret_cast<uint32_t*>(scratch) + (size_t)row * N;
  uint32_t* keys2 = reinterpret_cast<uint32_t*>(scratch) + total + (size_t)row * N;
  uint8_t* valid = scratch + 8 * (size_t)total + (size_t)row * N;
  const float* s = scores + (size_t)row * N;
  const int32_t* id = ids ? ids + (size_t)row * N : nullptr;

  // every call rewrites the whole row region it reads: no state carries over
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    keys[n] = order_key(s[n]);
    keys2[n] = 0xffffffffu - (uint32_t)(id ? id[n] : n);
    valid[n] = 0;
  }
  __syncthreads();

  const bool all = k >= N, none = k <= 0;
  uint32_t T = 0, T2 = 0;
  if (!all && !none) {
    int need = 0;
    T = row_radix_select(keys, nullptr, N, k, hist, sh, &need);
    int eq = 0;
    for (int n = threadIdx.x; n < N; n += blockDim.x) {
      const bool isT = __ldcg(keys + n) == T;
      valid[n] = isT;
      eq += isT;
    }
    for (int o = 16; o > 0; o >>= 1) eq += __shfl_xor_sync(0xffffffffu, eq, o);
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = eq;
    __syncthreads();
    if (threadIdx.x == 0) {
      int t = 0;
      for (int q = 0; q < (int)(blockDim.x >> 5); ++q) t += wsum[q];
      sh[0] = t;
    }
    __syncthreads();
    const int eq_total = sh[0];
    __syncthreads();
    if (need < eq_total) {
      int dummy = 0;
      T2 = row_radix_select(keys2, valid, N, need, hist, sh, &dummy);
    }
  }
  // compact the kept columns in ascending order.  Strictly kept: a larger
  // score, or the threshold score with a smaller id than the threshold id.
  // Entries equal to the threshold in score and id ("tied") fill the rest,
  // k - (strictly kept), in ascending column order.
  const int per = (N + blockDim.x - 1) / blockDim.x;
  const int n0 = min(N, (int)threadIdx.x * per), n1 = min(N, n0 + per);
  auto strict = [&](uint32_t a, uint32_t b2) { return all || a > T || (a == T && b2 > T2); };
  auto tied = [&](uint32_t a, uint32_t b2) { return !all && a == T && b2 == T2; };
  int cs = 0, ct = 0;
  for (int n = n0; n < n1; ++n) {
    const uint32_t a = __ldcg(keys + n), b2 = __ldcg(keys2 + n);
    cs += strict(a, b2);
    ct += tied(a, b2);
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (int)(blockDim.x >> 5);
  int is = cs, it = ct;
  for (int o = 1; o < 32; o <<= 1) {
    const int vs = __shfl_up_sync(0xffffffffu, is, o);
    const int vt = __shfl_up_sync(0xffffffffu, it, o);
    if (lane >= o) {
      is += vs;
      it += vt;
    }
  }
  __syncthreads();
  if (lane == 31) {
    wsum[wid] = is;
    wsum2[wid] = it;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int rs = 0, rt = 0;
    for (int q = 0; q < nw; ++q) {
      const int vs = wsum[q], vt = wsum2[q];
      wsum[q] = rs;
      wsum2[q] = rt;
      rs += vs;
      rt += vt;
    }
    sh[0] = rs;   // strictly kept in the row
  }
  __syncthreads();
  const int take = k - sh[0];
  int ps = wsum[wid] + is - cs, pt = wsum2[wid] + it - ct;
  for (int n = n0; n < n1; ++n) {
    const uint32_t a = __ldcg(keys + n), b2 = __ldcg(keys2 + n);
    if (strict(a, b2)) {
      const int at = ps + min(pt, take);
      if (at < k) kept[(size_t)row * k + at] = n;
      ++ps;
    } else if (tied(a, b2)) {
      if (pt < take) kept[(size_t)row * k + ps + pt] = n;
      ++pt;
    }
  }
}

// Device address of the scratch array for the current device, looked up once.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_READER_ECUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return MOE_READER_EINVAL;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_ready[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess || p == nullptr)
      return MOE_READER_ECUDA;
    g_scratch_ptr[dev] = p;
    g_scratch_ready[dev] = true;
  }
  *out = g_scratch_ptr[dev];
  return MOE_READER_OK;
}

}  // namespace

extern "C" int moe_reader_topk_noalloc(const float* scores, const int32_t* ids, int32_t rows,
                                       int32_t cols, int32_t k, int32_t* kept, void* stream) {
  if (rows < 0 || cols < 0 || k < 0 || k > cols) return MOE_READER_EINVAL;
  if (rows == 0 || k == 0) return MOE_READER_OK;
  if (!scores || !kept) return MOE_READER_EINVAL;
  if ((long long)rows * cols > kNoAllocMaxElems) return MOE_READER_ETOOBIG;
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != MOE_READER_OK) return st;
  topk_noalloc_kernel<<<rows, 1024, 0, static_cast<cudaStream_t>(stream)>>>(
      scores, ids, cols, k, kept, static_cast<unsigned char*>(scratch),
      (long long)rows * cols);
  return cudaGetLastError() == cudaSuccess ? MOE_READER_OK : MOE_READER_ECUDA;
}
