// Decode kernels of the channel reader ("Channel Selection for
// Mixture-of-Experts Decoding Needs No Calibration Data", Chinese summary
// page, 方法步骤详情 decode steps (1)-(4) and 核心方法; Korean summary page,
// 어떻게 쓰나).
//
//   rotate_kernel   Rx per 128-block (fp32 Sylvester butterfly of sigma*x) and
//                   the c largest-|Rx| coordinates per block; routing checks
//   screen_kernel   ghat/vhat partial sums per (token, expert, block) from the
//                   2-bit codes of the screened coordinates, scaled by alpha
//   topk_kernel     s_j = w_j ||d_j|| |phi(ghat_j) vhat_j|; exact top-k over all
//                   routed channels by radix select (ties -> lower e*I + i)
//   exact_kernel    kept channels: a_j from native BF16 g_j, v_j and fp32 x;
//                   skipped channels: recovery partials sum w_j p_j b_j
//   out_kernel      y = sum_K w_j a_j Dt_j + U c  (sector-wide column slices)
#include "device_util.cuh"
#include "internal.cuh"

namespace mr {
namespace {

// ---------------------------------------------------------------------------
// rotate_kernel: one warp per (token t, block b).  Lane l holds coordinates
// l + 32 s (s = 0..3).  Butterfly strides 1..16 across lanes, then 32 and 64
// in the lane: each pair (i, i+h) becomes (a + b, a - b) in fp32, the order
// that fixes the selection decision.  Rx = z / sqrt(128) (fp32).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128)
rotate_kernel(Dims d, int B, const float* __restrict__ x, const int32_t* __restrict__ ids_in,
              const float* __restrict__ w_in, const int8_t* __restrict__ sigma,
              float* __restrict__ rx, uint32_t* __restrict__ mask, int32_t* __restrict__ ids_ws,
              float* __restrict__ w_ws, uint32_t* __restrict__ err) {
  const int gwarp = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gwarp >= B * d.nb) return;
  const int t = gwarp / d.nb, b = gwarp % d.nb;

  // routing checks and sanitised copies (one warp per token)
  if (b == 0) {
    for (int s = lane; s < d.topk; s += 32) {
      int e = ids_in[t * d.topk + s];
      const float wv = w_in[t * d.topk + s];
      uint32_t bits = 0;
      if (e < 0 || e >= d.E) {
        bits |= kErrExpertRange;
        e = 0;
      }
      for (int s2 = 0; s2 < s; ++s2)
        if (ids_in[t * d.topk + s2] == ids_in[t * d.topk + s]) bits |= kErrExpertDup;
      if (!(wv >= 0.f) || !isfinite(wv)) bits |= kErrWeight;
      if (bits) atomicOr(err, bits);
      ids_ws[t * d.topk + s] = e;
      w_ws[t * d.topk + s] = wv;
    }
  }

  float u[4];
  bool bad = false;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int col = b * kBlock + lane + 32 * s;
    const float xv = col < d.H ? x[(size_t)t * d.H + col] : 0.f;
    bad |= !isfinite(xv);
    u[s] = sigma[col] < 0 ? -xv : xv;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(err, kErrXNonFinite);
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const float o = __shfl_xor_sync(0xffffffffu, u[s], h);
      u[s] = (lane & h) ? __fsub_rn(o, u[s]) : __fadd_rn(u[s], o);
    }
  }
  {
    float a0 = u[0], a1 = u[1], a2 = u[2], a3 = u[3];
    u[0] = __fadd_rn(a0, a1); u[1] = __fsub_rn(a0, a1);
    u[2] = __fadd_rn(a2, a3); u[3] = __fsub_rn(a2, a3);
    a0 = u[0]; a1 = u[1]; a2 = u[2]; a3 = u[3];
    u[0] = __fadd_rn(a0, a2); u[2] = __fsub_rn(a0, a2);
    u[1] = __fadd_rn(a1, a3); u[3] = __fsub_rn(a1, a3);
  }
  float m[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) m[s] = fabsf(u[s]);
  // rank of each coordinate: how many coordinates beat it (larger |z|, or equal and lower index)
  int rank[4] = {0, 0, 0, 0};
  for (int src = 0; src < 32; ++src) {
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2) {
      const float o = __shfl_sync(0xffffffffu, m[s2], src);
      const int oi = src + 32 * s2;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int mi = lane + 32 * s;
        rank[s] += (o > m[s]) || (o == m[s] && oi < mi);
      }
    }
  }
  const float inv = 0.08838834764831845f;   // 1/sqrt(128) rounded to fp32
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const unsigned sel = __ballot_sync(0xffffffffu, rank[s] < d.c);
    if (lane == 0) mask[((size_t)t * d.nb + b) * 4 + s] = sel;
    rx[(size_t)t * d.Hp + b * kBlock + lane + 32 * s] = u[s] * inv;
  }
}

// ---------------------------------------------------------------------------
// screen_kernel: one CTA per (token t, slot, block b).  Thread (q, j): word j
// of the coordinate record (j < I/16: gate run, else up run; 16 channels per
// 32-bit word), coordinate group q takes every Q-th screened coordinate.
// A 2-bit code shifted to bits 31:30 and masked is the fp32 value 2t (code
// 0b01 -> +2, 0b11 -> -2, 0b00 -> 0), so acc += (2t) * (r/2) is exact.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
screen_kernel(Dims d, int Q, const uint8_t* __restrict__ codes, const __half* __restrict__ scales,
              const float* __restrict__ rx, const uint32_t* __restrict__ mask,
              const int32_t* __restrict__ ids, float* __restrict__ partial) {
  extern __shared__ float red[];          // [Q][W*16]
  __shared__ int clist[kBlock];
  __shared__ float rlist[kBlock];
  const int b = blockIdx.x % d.nb;
  const int ts = blockIdx.x / d.nb;       // t * topk + slot
  const int t = ts / d.topk;
  const int e = ids[ts];
  const int W = d.I / 8;                  // words per coordinate record (gate + up)
  const int j = threadIdx.x % W;
  const int q = threadIdx.x / W;

  const uint32_t* mk = mask + ((size_t)t * d.nb + b) * 4;
  for (int c = threadIdx.x; c < kBlock; c += blockDim.x) {
    const uint32_t word = mk[c >> 5];
    if ((word >> (c & 31)) & 1u) {
      int pos = __popc(word & ((1u << (c & 31)) - 1u));
      for (int w2 = 0; w2 < (c >> 5); ++w2) pos += __popc(mk[w2]);
      clist[pos] = c;
      rlist[pos] = 0.5f * rx[(size_t)t * d.Hp + b * kBlock + c];
    }
  }
  __syncthreads();
  const int nsel = d.c;

  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  if (q < Q) {
    const int half = d.I / 16;
    const size_t run_off = j < half ? (size_t)j * 4 : (size_t)d.S + (size_t)(j - half) * 4;
    const uint8_t* base = codes + (((size_t)e * d.nb + b) * kBlock) * 2 * d.S + run_off;
    for (int p = q; p < nsel; p += Q) {
      // a non-finite x can leave the mask without exactly c bits: keep the
      // coordinate inside the block whatever the list holds
      const int c = clist[p] & (kBlock - 1);
      const float r = rlist[p];
      const uint32_t w = ldg_stream1(reinterpret_cast<const uint32_t*>(base + (size_t)c * 2 * d.S));
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float tv = __uint_as_float((w << (30 - 2 * k)) & 0xC0000000u);
        acc[k] = fmaf(tv, r, acc[k]);
      }
    }
  }
  const int WC = W * 16;
  if (q < Q) {
#pragma unroll
    for (int k = 0; k < 16; ++k) red[q * WC + j * 16 + k] = acc[k];
  }
  __syncthreads();
  // reduce over q and scale: channel slot (j, k) -> gv = j / (I/16), i = (j % (I/16)) * 16 + k
  const __half* sc = scales + ((size_t)e * d.nb + b) * 2 * d.I;
  float* out = partial + (((size_t)ts * d.nb + b) * 2) * d.I;
  for (int o = threadIdx.x; o < WC; o += blockDim.x) {
    float s = 0.f;
    for (int qq = 0; qq < Q; ++qq) s += red[qq * WC + o];
    const int jj = o / 16, k = o % 16;
    const int half = d.I / 16;
    const int gv = jj / half;
    const int i = (jj % half) * 16 + k;
    out[gv * d.I + i] = s * __half2float(sc[gv * d.I + i]);
  }
}

// ---------------------------------------------------------------------------
// topk_kernel: one CTA (1024 threads) per token.  Keys are the fp32 bits of
// s (s >= 0, so unsigned order = numeric order).  Radix select (4 x 8 bits)
// finds the k-th largest key T; keys above T are kept, and among keys equal to
// T the lowest global ids e*I + i are kept (second radix select on ~id).
// ---------------------------------------------------------------------------
__device__ uint32_t radix_select_desc(const uint32_t* keys, const uint8_t* valid, int N, int kth,
                                      int* hist, int* shared_out, int* remaining_out) {
  // returns the kth-largest key (1-based) among valid entries; *remaining_out =
  // how many entries equal to it are needed to reach kth
  uint32_t prefix = 0, pmask = 0;
  int remaining = kth;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int n = threadIdx.x; n < N; n += blockDim.x) {
      if (valid && !valid[n]) continue;
      const uint32_t kk = keys[n];
      if ((kk & pmask) == prefix) atomicAdd(&hist[(kk >> shift) & 255u], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // suffix scan from digit 255 down, 8 digits per lane
      const int lane = threadIdx.x;
      int local[8];
      int tot = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        local[u] = hist[255 - (lane * 8 + u)];
        tot += local[u];
      }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int before = incl - tot;   // count of digits above this lane's first digit
      int found = -1, rem = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (found < 0 && before + local[u] >= remaining) {
          found = 255 - (lane * 8 + u);
          rem = remaining - before;
        }
        before += local[u];
      }
      const unsigned bal = __ballot_sync(0xffffffffu, found >= 0);
      const int first = __ffs(bal) - 1;
      const int fd = __shfl_sync(0xffffffffu, found, first);
      const int fr = __shfl_sync(0xffffffffu, rem, first);
      if (lane == 0) {
        shared_out[0] = fd;
        shared_out[1] = fr;
      }
    }
    __syncthreads();
    const int digit = shared_out[0];
    remaining = shared_out[1];
    prefix |= (uint32_t)digit << shift;
    pmask |= 255u << shift;
    __syncthreads();
  }
  *remaining_out = remaining;
  return prefix;
}

__global__ void __launch_bounds__(1024)
topk_kernel(Dims d, int k, const float* __restrict__ partial, const int32_t* __restrict__ ids,
            const float* __restrict__ wts, const float* __restrict__ dnorm,
            float* __restrict__ ghat, float* __restrict__ vhat, float* __restrict__ pout,
            float* __restrict__ score, uint32_t* __restrict__ keptbits,
            int32_t* __restrict__ kept) {
  extern __shared__ uint32_t keys[];      // [N] then [N] tie keys, [N] bytes valid
  uint32_t* keys2 = keys + d.N;
  uint8_t* valid = reinterpret_cast<uint8_t*>(keys2 + d.N);
  __shared__ int hist[256];
  __shared__ int sout[2];
  __shared__ int wsum[32];
  const int t = blockIdx.x;
  const int N = d.N;

  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    const int slot = n / d.I, i = n % d.I;
    const float* pg = partial + (((size_t)(t * d.topk + slot) * d.nb) * 2) * d.I + i;
    float g = 0.f, v = 0.f;
    for (int b = 0; b < d.nb; ++b) {
      g += pg[(size_t)b * 2 * d.I];
      v += pg[(size_t)b * 2 * d.I + d.I];
    }
    const int e = ids[t * d.topk + slot];
    const float p = silu_f(g) * v;
    const float s = wts[t * d.topk + slot] * dnorm[(size_t)e * d.I + i] * fabsf(p);
    const size_t o = (size_t)t * N + n;
    ghat[o] = g;
    vhat[o] = v;
    pout[o] = p;
    score[o] = s;
    keys[n] = __float_as_uint(s);
  }
  __syncthreads();

  uint32_t T = 0, T2 = 0;
  int need = 0;
  const bool all = k >= N, none = k <= 0;
  if (!all && !none) {
    T = radix_select_desc(keys, nullptr, N, k, hist, sout, &need);
    // ties at T: keep the `need` lowest global ids
    int eq = 0;
    for (int n = threadIdx.x; n < N; n += blockDim.x) {
      const bool isT = keys[n] == T;
      valid[n] = isT;
      const int slot = n / d.I, i = n % d.I;
      keys2[n] = 0xffffffffu - (uint32_t)(ids[t * d.topk + slot] * d.I + i);
      eq += isT;
    }
    __syncthreads();
    // count of equal keys (block reduction)
    eq = warp_sum_i(eq);
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = eq;
    __syncthreads();
    if (threadIdx.x == 0) {
      int tot = 0;
      for (int q = 0; q < (int)(blockDim.x >> 5); ++q) tot += wsum[q];
      sout[0] = tot;
    }
    __syncthreads();
    const int eq_total = sout[0];
    __syncthreads();
    if (need < eq_total) {
      int dummy = 0;
      T2 = radix_select_desc(keys2, valid, N, need, hist, sout, &dummy);
    } else {
      T2 = 0;   // keep every tied key
    }
  }
  // kept flags, bitmap and the ascending list of kept n
  const int per = (N + blockDim.x - 1) / blockDim.x;
  const int n0 = threadIdx.x * per;
  const int n1 = min(N, n0 + per);
  int cnt = 0;
  for (int n = n0; n < n1; ++n) {
    bool kp;
    if (all) kp = true;
    else if (none) kp = false;
    else kp = keys[n] > T || (keys[n] == T && keys2[n] >= T2);
    cnt += kp;
  }
  // exclusive scan of cnt over threads
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  __syncthreads();
  if (lane == 31) wsum[wid] = incl;
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int q = 0; q < (int)(blockDim.x >> 5); ++q) {
      const int v = wsum[q];
      wsum[q] = run;
      run += v;
    }
  }
  __syncthreads();
  int pos = wsum[wid] + incl - cnt;
  for (int n = n0; n < n1; ++n) {
    bool kp;
    if (all) kp = true;
    else if (none) kp = false;
    else kp = keys[n] > T || (keys[n] == T && keys2[n] >= T2);
    if (kp) kept[(size_t)t * N + pos++] = n;
  }
  // bitmap: one word per 32 channels
  for (int wdx = threadIdx.x; wdx < N / 32; wdx += blockDim.x) {
    uint32_t bits = 0;
    for (int u = 0; u < 32; ++u) {
      const int n = wdx * 32 + u;
      bool kp;
      if (all) kp = true;
      else if (none) kp = false;
      else kp = keys[n] > T || (keys[n] == T && keys2[n] >= T2);
      bits |= (uint32_t)kp << u;
    }
    keptbits[(size_t)t * (N / 32) + wdx] = bits;
  }
}

// ---------------------------------------------------------------------------
// exact_kernel: warps [0, B*k) take kept channels (a_j from native rows),
// warps [B*k, B*k + B*N/64) take 64-channel recovery chunks.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
exact_kernel(Dims d, int B, int k, const float* __restrict__ x, const __nv_bfloat16* __restrict__ G,
             const __nv_bfloat16* __restrict__ V, const int32_t* __restrict__ ids,
             const float* __restrict__ wts, const int32_t* __restrict__ kept,
             const uint32_t* __restrict__ keptbits, const float* __restrict__ p,
             const __half* __restrict__ bco, float* __restrict__ wa, float* __restrict__ cpart) {
  const long long gw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long nk = (long long)B * k;
  const int chunks = d.N / 64;
  if (gw < nk) {
    const int t = (int)(gw / k), qi = (int)(gw % k);
    const int n = kept[(size_t)t * d.N + qi];
    const int slot = n / d.I, i = n % d.I;
    const int e = ids[t * d.topk + slot];
    const uint4* g4 = reinterpret_cast<const uint4*>(G + ((size_t)e * d.I + i) * d.H);
    const uint4* v4 = reinterpret_cast<const uint4*>(V + ((size_t)e * d.I + i) * d.H);
    const float4* x4 = reinterpret_cast<const float4*>(x + (size_t)t * d.H);
    float sg = 0.f, sv = 0.f;
    for (int h8 = lane; h8 < d.H / 8; h8 += 32) {
      const uint4 gq = ldg_stream(g4 + h8);
      const uint4 vq = ldg_stream(v4 + h8);
      const float4 xa = x4[2 * h8], xb = x4[2 * h8 + 1];
      sg = fmaf(bf16_lo(gq.x), xa.x, sg); sg = fmaf(bf16_hi(gq.x), xa.y, sg);
      sg = fmaf(bf16_lo(gq.y), xa.z, sg); sg = fmaf(bf16_hi(gq.y), xa.w, sg);
      sg = fmaf(bf16_lo(gq.z), xb.x, sg); sg = fmaf(bf16_hi(gq.z), xb.y, sg);
      sg = fmaf(bf16_lo(gq.w), xb.z, sg); sg = fmaf(bf16_hi(gq.w), xb.w, sg);
      sv = fmaf(bf16_lo(vq.x), xa.x, sv); sv = fmaf(bf16_hi(vq.x), xa.y, sv);
      sv = fmaf(bf16_lo(vq.y), xa.z, sv); sv = fmaf(bf16_hi(vq.y), xa.w, sv);
      sv = fmaf(bf16_lo(vq.z), xb.x, sv); sv = fmaf(bf16_hi(vq.z), xb.y, sv);
      sv = fmaf(bf16_lo(vq.w), xb.z, sv); sv = fmaf(bf16_hi(vq.w), xb.w, sv);
    }
    sg = warp_sum(sg);
    sv = warp_sum(sv);
    if (lane == 0) wa[(size_t)t * d.N + qi] = wts[t * d.topk + slot] * silu_f(sg) * sv;
    return;
  }
  const long long rw = gw - nk;
  if (rw >= (long long)B * chunks) return;
  const int t = (int)(rw / chunks), ch = (int)(rw % chunks);
  const int n0 = ch * 64;
  const int slot = n0 / d.I;
  const int e = ids[t * d.topk + slot];
  const float wv = wts[t * d.topk + slot];
  const uint32_t kb0 = keptbits[(size_t)t * (d.N / 32) + ch * 2];
  const uint32_t kb1 = keptbits[(size_t)t * (d.N / 32) + ch * 2 + 1];
  float a0 = 0.f, a1 = 0.f;
  for (int u = 0; u < 64; ++u) {
    const uint32_t kb = u < 32 ? kb0 : kb1;
    if ((kb >> (u & 31)) & 1u) continue;
    const int n = n0 + u;
    const int i = n % d.I;
    const float coef = wv * p[(size_t)t * d.N + n];
    const __half* brow = bco + ((size_t)e * d.I + i) * d.r;
    if (lane < d.r) a0 = fmaf(coef, __half2float(brow[lane]), a0);
    if (lane + 32 < d.r) a1 = fmaf(coef, __half2float(brow[lane + 32]), a1);
  }
  float* cp = cpart + ((size_t)t * chunks + ch) * d.r;
  if (lane < d.r) cp[lane] = a0;
  if (lane + 32 < d.r) cp[lane + 32] = a1;
}

// ---------------------------------------------------------------------------
// out_kernel: one CTA per 16-column slice h0..h0+15 (one 32-byte sector of
// each transposed down row).  Thread (rg, half): kept rows rg, rg+128, ...;
// 8 columns each.  y = sum_K (w a)_j Dt_j + U c, c = sum over recovery chunks.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
out_kernel(Dims d, int B, int k, const __nv_bfloat16* __restrict__ Dt,
           const int32_t* __restrict__ ids, const int32_t* __restrict__ kept,
           const float* __restrict__ wa, const float* __restrict__ cpart,
           const __half* __restrict__ U, float* __restrict__ y) {
  __shared__ float red[128][17];
  __shared__ float cvec[kMaxRank];
  const int h0 = blockIdx.x * 16;
  const int rg = threadIdx.x >> 1, hf = threadIdx.x & 1;
  const int chunks = d.N / 64;
  for (int t = 0; t < B; ++t) {
    float acc[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[u] = 0.f;
    const int hh = h0 + hf * 8;
    if (hh < d.H) {
      for (int q = rg; q < k; q += 128) {
        const int n = kept[(size_t)t * d.N + q];
        const int slot = n / d.I, i = n % d.I;
        const int e = ids[t * d.topk + slot];
        const float c = wa[(size_t)t * d.N + q];
        const uint4 dq = ldg_stream(reinterpret_cast<const uint4*>(Dt + ((size_t)e * d.I + i) * d.H + hh));
        acc[0] = fmaf(c, bf16_lo(dq.x), acc[0]); acc[1] = fmaf(c, bf16_hi(dq.x), acc[1]);
        acc[2] = fmaf(c, bf16_lo(dq.y), acc[2]); acc[3] = fmaf(c, bf16_hi(dq.y), acc[3]);
        acc[4] = fmaf(c, bf16_lo(dq.z), acc[4]); acc[5] = fmaf(c, bf16_hi(dq.z), acc[5]);
        acc[6] = fmaf(c, bf16_lo(dq.w), acc[6]); acc[7] = fmaf(c, bf16_hi(dq.w), acc[7]);
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) red[rg][hf * 8 + u] = acc[u];
    // recovery vector c for token t
    if (threadIdx.x < d.r) {
      float s = 0.f;
      if (k < d.N)
        for (int ch = 0; ch < chunks; ++ch) s += cpart[((size_t)t * chunks + ch) * d.r + threadIdx.x];
      cvec[threadIdx.x] = s;
    }
    __syncthreads();
    if (threadIdx.x < 16) {
      const int h = h0 + threadIdx.x;
      float s = 0.f;
      for (int q = 0; q < 128; ++q) s += red[q][threadIdx.x];
      if (h < d.H) {
        if (k < d.N)
          for (int j = 0; j < d.r; ++j) s = fmaf(__half2float(U[(size_t)h * d.r + j]), cvec[j], s);
        y[(size_t)t * d.H + h] = s;
      }
    }
    __syncthreads();
  }
}

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

int screen_groups(const Dims& d) {
  const int W = d.I / 8;
  int Q = 1024 / W;
  if (Q > 8) Q = 8;
  if (Q < 1) Q = 1;
  return Q;
}

}  // namespace

cudaError_t launch_decode(const moe_reader& h, const float* x, int B, const int32_t* ids,
                          const float* w, int k, float* y, cudaStream_t s,
                          const cudaEvent_t* ev) {
  const Dims& d = h.d;
  const Workspace& ws = h.ws;
  cudaError_t err;
  // Inside stream capture a plain event record is only a dependency marker;
  // the External flag makes it an event-record node of the graph.
  unsigned int rec_flags = cudaEventRecordDefault;
  if (ev) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if ((err = cudaStreamIsCapturing(s, &cs)) != cudaSuccess) return err;
    if (cs == cudaStreamCaptureStatusActive) rec_flags = cudaEventRecordExternal;
  }
#define MR_MARK(i) \
  if (ev && (err = cudaEventRecordWithFlags(ev[i], s, rec_flags)) != cudaSuccess) return err;
  MR_MARK(0)
  const int rot_warps = B * d.nb;
  rotate_kernel<<<(rot_warps + 3) / 4, 128, 0, s>>>(d, B, x, ids, w, h.p.sigma, ws.rx, ws.mask,
                                                    ws.ids, ws.w, ws.err);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  MR_MARK(1)

  const int Q = screen_groups(d);
  const int W = d.I / 8;
  const size_t ssm = (size_t)Q * W * 16 * sizeof(float);
  screen_kernel<<<B * d.topk * d.nb, W * Q, ssm, s>>>(d, Q, h.p.codes, h.p.scales, ws.rx, ws.mask,
                                                      ws.ids, ws.partial);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  MR_MARK(2)

  const size_t tsm = (size_t)d.N * 9;
  topk_kernel<<<B, 1024, tsm, s>>>(d, k, ws.partial, ws.ids, ws.w, h.p.dnorm, ws.ghat, ws.vhat,
                                   ws.p, ws.score, ws.keptbits, ws.kept);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  MR_MARK(3)

  const long long warps = (long long)B * k + (long long)B * (d.N / 64);
  exact_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(d, B, k, x, h.G, h.V, ws.ids, ws.w,
                                                           ws.kept, ws.keptbits, ws.p, h.p.b,
                                                           ws.wa, ws.cpart);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  MR_MARK(4)

  out_kernel<<<(d.H + 15) / 16, 256, 0, s>>>(d, B, k, h.p.Dt, ws.ids, ws.kept, ws.wa, ws.cpart,
                                              h.p.U, y);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  MR_MARK(5)
#undef MR_MARK
  return cudaSuccess;
}

// Dynamic shared memory limits are per kernel, not per handle: only ever raise them.
template <typename K>
cudaError_t raise_smem_limit(K kernel, size_t bytes) {
  cudaFuncAttributes fa;
  cudaError_t err = cudaFuncGetAttributes(&fa, kernel);
  if (err != cudaSuccess) return err;
  if ((size_t)fa.maxDynamicSharedSizeBytes >= bytes) return cudaSuccess;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

cudaError_t configure_decode_kernels(const Dims& d) {
  const int Q = screen_groups(d);
  const int W = d.I / 8;
  cudaError_t err = raise_smem_limit(screen_kernel, (size_t)Q * W * 16 * sizeof(float));
  if (err != cudaSuccess) return err;
  return raise_smem_limit(topk_kernel, (size_t)d.N * 9);
}

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
