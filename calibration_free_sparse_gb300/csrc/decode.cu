// Decode of the channel reader as ONE persistent cooperative kernel per call
// ("Channel Selection for Mixture-of-Experts Decoding Needs No Calibration
// Data", Chinese summary page, 方法步骤详情 decode steps (1)-(4) and 核心方法;
// Korean summary page, 어떻게 쓰나).
//
// One CTA per SM, all co-resident (cooperative launch).  The phases hand work
// to each other through counters and flags in global memory instead of
// kernel boundaries; every wait is bounded (about one second of globaltimer),
// after which the CTA raises the timeout bit and the abort flag and leaves.
//
//   phase 0  rotate x per (token, 128-block): fp32 Sylvester butterfly of
//            sigma*x, the c largest |Rx| coordinates (ties -> lower index),
//            routing checks; sets rot_flag[t][b]
//   phase 1  screen unit per (token, expert slot, block): the 2-bit codes of
//            the screened coordinates, alpha-scaled block partials of ghat and
//            vhat.  The last unit of a (token, slot) sums the block partials in
//            block order and scores the slot's channels,
//            s = w ||d|| |phi(ghat) vhat|; the last slot of a token runs the
//            exact top-k over the token's N channels (radix select on the fp32
//            bits, ties -> lower e*I + i) and sets tok_flag[t]
//   phase 2  warp items: kept channels (a_j = phi(g_j.x)(v_j.x) from native
//            BF16 rows, fp32 x) and 64-channel recovery chunks
//            (sum w_j p_j b_j over skipped channels)
//   phase 3  output slices of 16 columns: y = sum_K w_j a_j Dt_j + U c
#include "device_util.cuh"
#include "internal.cuh"

namespace mr {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kAhead = 8;              // code words a thread loads before using them
constexpr int kMaxGroups = 16;         // coordinate groups of a screen unit
constexpr unsigned long long kWaitNs = 1000000000ull;

struct Params {
  Dims d;
  int B, k;
  const float* x;
  const int32_t* ids_in;
  const float* w_in;
  float* y;
  const int8_t* sigma;
  const uint8_t* codes;
  const __half* scales;
  const float* dnorm;
  const __nv_bfloat16* G;
  const __nv_bfloat16* V;
  const __nv_bfloat16* Dt;
  const __half* U;
  const __half* bco;
  int32_t* ids_ws;
  float* w_ws;
  float* rx;
  uint32_t* mask;
  float* partial;
  float* ghat;
  float* vhat;
  float* p;
  float* score;
  uint32_t* keptbits;
  int32_t* kept;
  int32_t* rowoff;
  float* wa;
  float* cvec;                  // [Bmax][r] recovery vectors, accumulated atomically
  unsigned long long* stamps;   // [grid][5] phase timestamps, or null
  uint32_t* sync;
  uint32_t* err;
  int Q;    // coordinate groups of a screen unit
  int W8;   // 8-byte code words per coordinate record (gate run + up run)
};

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint2 ldg_nc2(const void* p) {
  uint2 r;
  asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 ldg_nc4(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// Wait (one thread) until *flag >= target.  false: timed out or aborted.
__device__ bool wait_at_least(const uint32_t* flag, uint32_t target, uint32_t* abort_flag,
                              uint32_t* err) {
  if (ld_acquire(flag) >= target) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (ld_acquire(flag) >= target) return true;
    if (ld_acquire(abort_flag)) return false;
    if (globaltimer() - t0 > kWaitNs) {
      atomicOr(err, kErrTimeout);
      atomicExch(abort_flag, 1u);
      return false;
    }
    __nanosleep(64);
  }
}

// Offsets (in uint32) of the synchronisation area, fixed per handle.
struct SyncOff {
  int rot, slot, tok, flag, total;
};
__host__ __device__ inline SyncOff sync_offsets(const Dims& d) {
  SyncOff o;
  o.rot = 16;
  o.slot = o.rot + d.Bmax * d.nb;
  o.tok = o.slot + d.Bmax * d.topk;
  o.flag = o.tok + d.Bmax;
  o.total = o.flag + d.Bmax;
  return o;
}
constexpr int kSyncDone = 0, kSyncExact = 1, kSyncAbort = 2, kSyncNext = 3;

// ------------------------------- phase 0 -----------------------------------
__device__ void rotate_item(const Params& P, int t, int b, int lane) {
  const Dims& d = P.d;
  uint32_t* err = P.err;
  if (b == 0) {
    for (int s = lane; s < d.topk; s += 32) {
      int e = P.ids_in[t * d.topk + s];
      const float wv = P.w_in[t * d.topk + s];
      uint32_t bits = 0;
      if (e < 0 || e >= d.E) {
        bits |= kErrExpertRange;
        e = 0;
      }
      for (int s2 = 0; s2 < s; ++s2)
        if (P.ids_in[t * d.topk + s2] == P.ids_in[t * d.topk + s]) bits |= kErrExpertDup;
      if (!(wv >= 0.f) || !isfinite(wv)) bits |= kErrWeight;
      if (bits) atomicOr(err, bits);
      P.ids_ws[t * d.topk + s] = e;
      P.w_ws[t * d.topk + s] = wv;
    }
    for (int j = lane; j < d.r; j += 32) P.cvec[(size_t)t * d.r + j] = 0.f;
  }
  float u[4];
  bool bad = false;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int col = b * kBlock + lane + 32 * s;
    const float xv = col < d.H ? P.x[(size_t)t * d.H + col] : 0.f;
    bad |= !isfinite(xv);
    u[s] = P.sigma[col] < 0 ? -xv : xv;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(err, kErrXNonFinite);
  // Sylvester butterfly, strides 1, 2, ..., 64; pair (i, i+h) -> (a + b, a - b) in fp32
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
  // the c-th largest |z| by a bit search over its fp32 pattern, then ties by index
  uint32_t m[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) m[s] = __float_as_uint(fabsf(u[s]));
  uint32_t T = 0;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t cand = T | (1u << bit);
    int cnt = 0;
#pragma unroll
    for (int s = 0; s < 4; ++s) cnt += __popc(__ballot_sync(0xffffffffu, m[s] >= cand));
    if (cnt >= d.c) T = cand;
  }
  int gt = 0;
#pragma unroll
  for (int s = 0; s < 4; ++s) gt += __popc(__ballot_sync(0xffffffffu, m[s] > T));
  const int need = d.c - gt;
  const uint32_t below = (1u << lane) - 1u;
  int before = 0;
  const float inv = 0.08838834764831845f;   // 1/sqrt(128) rounded to fp32
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const uint32_t eqb = __ballot_sync(0xffffffffu, m[s] == T);
    const bool sel = m[s] > T || (m[s] == T && before + __popc(eqb & below) < need);
    before += __popc(eqb);
    const uint32_t word = __ballot_sync(0xffffffffu, sel);
    if (lane == 0) P.mask[((size_t)t * d.nb + b) * 4 + s] = word;
    P.rx[(size_t)t * d.Hp + b * kBlock + lane + 32 * s] = u[s] * inv;
  }
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    atomicExch(&P.sync[sync_offsets(d).rot + t * d.nb + b], 1u);
  }
}

// ------------------------------- top-k -------------------------------------
// k-th largest key among the entries keyfn accepts; per-warp histograms.
template <typename KeyFn>
__device__ uint32_t cta_radix_select(int N, int kth, KeyFn keyfn, int* hist, int* sh, int* rem) {
  uint32_t prefix = 0, pmask = 0;
  int remaining = kth;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < kWarps * 256; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int n = threadIdx.x; n < N; n += kThreads) {
      uint32_t key;
      if (!keyfn(n, key)) continue;
      if ((key & pmask) == prefix) atomicAdd(&hist[warp * 256 + ((key >> shift) & 255u)], 1);
    }
    __syncthreads();
    if (threadIdx.x < 256) {
      int tot = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) tot += hist[w * 256 + threadIdx.x];
      hist[kWarps * 256 + threadIdx.x] = tot;
    }
    __syncthreads();
    if (warp == 0) {
      const int* totals = hist + kWarps * 256;
      int local[8];
      int tot = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        local[u] = totals[255 - (lane * 8 + u)];
        tot += local[u];
      }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int before = incl - tot, found = -1, r = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (found < 0 && before + local[u] >= remaining) {
          found = 255 - (lane * 8 + u);
          r = remaining - before;
        }
        before += local[u];
      }
      const unsigned bal = __ballot_sync(0xffffffffu, found >= 0);
      const int first = bal ? __ffs(bal) - 1 : 0;
      const int fd = __shfl_sync(0xffffffffu, found, first);
      const int fr = __shfl_sync(0xffffffffu, r, first);
      if (lane == 0) {
        sh[0] = fd < 0 ? 0 : fd;
        sh[1] = fr;
      }
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

constexpr int kDigitBits = 12;               // first histogram: key bits 30..19
constexpr int kBins = 1 << kDigitBits;
constexpr int kCandMax = 1024;               // candidates ranked exactly; more -> radix

__device__ __forceinline__ int key_digit(uint32_t key) { return (int)((key >> 19) & (kBins - 1)); }

// Shared-memory layout of the top-k step (offsets in bytes from smem).
__host__ __device__ inline size_t topk_smem_bytes(int N) {
  return (size_t)4 * N                       // keys
         + (size_t)(kWarps + 1) * 256 * 4    // histogram (4096 bins, or the radix rows)
         + (size_t)N                         // keep flags
         + (size_t)kCandMax * 12             // candidate keys, ids, ranks
         + 512;                              // scalars, warp sums, expert ids
}

__device__ void topk_token(const Params& P, int t, unsigned char* smem) {
  const Dims& d = P.d;
  const int N = d.N, k = P.k, I = d.I;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem);                      // [N]
  int* hist = reinterpret_cast<int*>(keys + N);                             // [(kWarps+1)*256]
  uint8_t* keep = reinterpret_cast<uint8_t*>(hist + (kWarps + 1) * 256);    // [N]
  uint32_t* ckey = reinterpret_cast<uint32_t*>(keep + ((N + 15) & ~15));    // [kCandMax]
  uint32_t* cgid = ckey + kCandMax;                                         // [kCandMax]
  int* crank = reinterpret_cast<int*>(cgid + kCandMax);                     // [kCandMax]
  int* sh = crank + kCandMax;                                               // [8]
  int* wsum = sh + 8;                                                       // [kWarps]
  int* eid = wsum + kWarps;                                                 // [topk]
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int s = threadIdx.x; s < d.topk; s += kThreads) eid[s] = __ldcg(P.ids_ws + t * d.topk + s);
  for (int n = threadIdx.x; n < N; n += kThreads)
    keys[n] = __float_as_uint(__ldcg(P.score + (size_t)t * N + n));
  for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = 0;
  if (threadIdx.x == 0) sh[2] = 0;
  __syncthreads();

  const bool all = k >= N, none = k <= 0;
  if (all || none) {
    for (int n = threadIdx.x; n < N; n += kThreads) keep[n] = all;
  } else {
    // 1. histogram of the 12-bit digit (keys spread over hundreds of bins)
    for (int n = threadIdx.x; n < N; n += kThreads) atomicAdd(&hist[key_digit(keys[n])], 1);
    __syncthreads();
    // 2. the digit D holding the k-th largest key: 8 digits per thread, from the top
    constexpr int kPer = kBins / kThreads;
    int cnt[kPer], tot = 0;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      cnt[u] = hist[kBins - 1 - (threadIdx.x * kPer + u)];
      tot += cnt[u];
    }
    int incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[wid] = incl;
    __syncthreads();
    int before = incl - tot;
    for (int w = 0; w < wid; ++w) before += wsum[w];
    if (before < k && before + tot >= k) {
      int above = before;
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        if (above + cnt[u] >= k) {
          sh[0] = kBins - 1 - (threadIdx.x * kPer + u);
          sh[1] = k - above;       // keys of digit D that are kept
          sh[3] = cnt[u];          // keys of digit D
          break;
        }
        above += cnt[u];
      }
    }
    __syncthreads();
    const int D = sh[0], need = sh[1], m = sh[3];
    if (m <= kCandMax) {
      // 3. the candidates (digit D) ranked exactly: larger key, then lower global id
      for (int n = threadIdx.x; n < N; n += kThreads) {
        const int dg = key_digit(keys[n]);
        keep[n] = dg > D;
        if (dg == D) {
          const int c = atomicAdd(&sh[2], 1);
          ckey[c] = keys[n] | 0u;
          cgid[c] = (uint32_t)(eid[n / I] * I + n % I);
          crank[c] = n;             // the channel for now; the rank below
        }
      }
      __syncthreads();
      // every (ci, cj) pair once, spread over the threads
      const int pairs = m * m;
      int* rk = hist;               // reuse: rank counters [m]
      for (int c = threadIdx.x; c < m; c += kThreads) rk[c] = 0;
      __syncthreads();
      for (int q = threadIdx.x; q < pairs; q += kThreads) {
        const int ci = q / m, cj = q - ci * m;
        const uint32_t ki = ckey[ci], kj = ckey[cj];
        if (kj > ki || (kj == ki && cgid[cj] < cgid[ci])) atomicAdd(&rk[ci], 1);
      }
      __syncthreads();
      for (int c = threadIdx.x; c < m; c += kThreads) keep[crank[c]] = rk[c] < need;
    } else {
      // degenerate spread (too many keys in one digit): full radix select
      int need2 = 0;
      const uint32_t T = cta_radix_select(
          N, k, [&](int n, uint32_t& key) { key = keys[n]; return true; }, hist, sh + 4, &need2);
      int eq = 0;
      for (int n = threadIdx.x; n < N; n += kThreads) eq += keys[n] == T;
      eq = warp_sum_i(eq);
      if (lane == 0) wsum[wid] = eq;
      __syncthreads();
      int eq_total = 0;
      for (int w = 0; w < kWarps; ++w) eq_total += wsum[w];
      __syncthreads();
      uint32_t T2 = 0;
      if (need2 < eq_total) {
        int dummy = 0;
        T2 = cta_radix_select(
            N, need2,
            [&](int n, uint32_t& key) {
              if (keys[n] != T) return false;
              key = 0xffffffffu - (uint32_t)(eid[n / I] * I + n % I);
              return true;
            },
            hist, sh + 4, &dummy);
      }
      for (int n = threadIdx.x; n < N; n += kThreads) {
        const uint32_t a = keys[n];
        keep[n] = a > T || (a == T && 0xffffffffu - (uint32_t)(eid[n / I] * I + n % I) >= T2);
      }
    }
  }
  __syncthreads();
  // 4. compaction in ascending n and the kept bitmap: warp w owns a contiguous
  //    range of whole 32-channel words; one ballot per word
  const int words = N / 32;
  const int wper = (words + kWarps - 1) / kWarps;
  const int w0 = wid * wper, w1 = min(words, w0 + wper);
  int mine = 0;
  for (int wd = w0; wd < w1; ++wd) mine += __popc(__ballot_sync(0xffffffffu, keep[wd * 32 + lane]));
  if (lane == 0) wsum[wid] = mine;
  __syncthreads();
  int pos = 0;
  for (int w = 0; w < wid; ++w) pos += wsum[w];
  const uint32_t below = (1u << lane) - 1u;
  for (int wd = w0; wd < w1; ++wd) {
    const int n = wd * 32 + lane;
    const uint32_t bal = __ballot_sync(0xffffffffu, keep[n]);
    if (keep[n]) {
      const int at = pos + __popc(bal & below);
      if (at < N) P.kept[(size_t)t * N + at] = n;
    }
    if (lane == 0) P.keptbits[(size_t)t * words + wd] = bal;
    pos += __popc(bal);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicExch(&P.sync[sync_offsets(d).flag + t], 1u);
  }
}

// ------------------------------- phase 1 -----------------------------------
// A screen unit runs on UT threads of the CTA: the whole CTA (UT = 512) when
// there are fewer units than CTAs, otherwise each half of the CTA (UT = 256)
// runs its own unit, synchronised by a named barrier, so two units' memory
// round trips overlap on every SM.
struct UnitCtx {
  int ut;              // thread index within the unit
  int UT;              // threads of the unit
  int bar;             // named barrier id (0 = __syncthreads)
  unsigned char* sm;   // this unit's shared memory
};

__device__ __forceinline__ void unit_sync(const UnitCtx& c) {
  if (c.UT == kThreads)
    __syncthreads();
  else
    asm volatile("bar.sync %0, %1;" ::"r"(c.bar), "r"(c.UT) : "memory");
}

__host__ __device__ inline int unit_groups(int W8, int UT) {
  int Q = UT / W8;
  if (Q > kMaxGroups) Q = kMaxGroups;
  return Q < 1 ? 1 : Q;
}

__host__ __device__ inline size_t unit_smem_bytes(int I, int Q) {
  const int Wp = (I / 16) | 1;
  return (size_t)4 * I + kBlock * 8 + 16 + (size_t)Q * 32 * Wp * 4;
}

// One (token, slot, block) unit: alpha-scaled block partials of ghat/vhat.
// false: the CTA must stop (timeout / abort).
__device__ bool screen_unit(const Params& P, int t, int slot, int b, const UnitCtx& cx) {
  const Dims& d = P.d;
  const SyncOff so = sync_offsets(d);
  const int ts = t * d.topk + slot;
  int e = P.ids_in[ts];
  if (e < 0 || e >= d.E) e = 0;
  const int I = d.I;
  // shared memory: alpha [2I] half, clist [128] int, rlist [128] float, flags [4], red [Q][32][Wp]
  __half* alpha = reinterpret_cast<__half*>(cx.sm);
  int* clist = reinterpret_cast<int*>(cx.sm + 4 * (size_t)I);
  float* rlist = reinterpret_cast<float*>(clist + kBlock);
  int* flags = reinterpret_cast<int*>(rlist + kBlock);
  float* red = reinterpret_cast<float*>(flags + 4);

  // alpha, the mask words and the rotation flag are requested together
  const __half* sc = P.scales + ((size_t)e * d.nb + b) * 2 * I;
  for (int i = cx.ut; i < I / 4; i += cx.UT)
    reinterpret_cast<uint4*>(alpha)[i] = ldg_nc4(reinterpret_cast<const uint4*>(sc) + i);
  if (cx.ut == 0)
    flags[0] = wait_at_least(P.sync + so.rot + t * d.nb + b, 1u, P.sync + kSyncAbort, P.err);
  unit_sync(cx);
  if (!flags[0]) return false;
  if (cx.ut < kBlock) {
    const int c = cx.ut;
    const uint32_t* mk = P.mask + ((size_t)t * d.nb + b) * 4;
    const uint4 mw = __ldcg(reinterpret_cast<const uint4*>(mk));
    const uint32_t words[4] = {mw.x, mw.y, mw.z, mw.w};
    const uint32_t word = words[c >> 5];
    if ((word >> (c & 31)) & 1u) {
      int pos = __popc(word & ((1u << (c & 31)) - 1u));
#pragma unroll
      for (int w2 = 0; w2 < 3; ++w2) pos += w2 < (c >> 5) ? __popc(words[w2]) : 0;
      if (pos < kBlock) {
        clist[pos] = c;
        rlist[pos] = 0.5f * __ldcg(P.rx + (size_t)t * d.Hp + b * kBlock + c);
      }
    }
  }
  unit_sync(cx);

  const int W8 = P.W8, Q = unit_groups(W8, cx.UT), Wp = W8 | 1;
  const int j = cx.ut % W8, q = cx.ut / W8;
  const int half = I / 32;                          // 8-byte words per run
  if (q < Q) {
    float acc[32];
#pragma unroll
    for (int u = 0; u < 32; ++u) acc[u] = 0.f;
    const size_t run_off = j < half ? (size_t)j * 8 : (size_t)d.S + (size_t)(j - half) * 8;
    const uint8_t* base = P.codes + (((size_t)e * d.nb + b) * kBlock) * 2 * d.S + run_off;
    for (int p0 = q; p0 < d.c; p0 += Q * kAhead) {
      uint2 wv[kAhead];
      float rv[kAhead];
#pragma unroll
      for (int u = 0; u < kAhead; ++u) {
        const int pp = p0 + u * Q;
        if (pp < d.c) {
          const int cc = clist[pp] & (kBlock - 1);
          wv[u] = ldg_nc2(base + (size_t)cc * 2 * d.S);
          rv[u] = rlist[pp];
        } else {
          wv[u] = make_uint2(0u, 0u);
          rv[u] = 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < kAhead; ++u) {
        // a 2-bit code moved to bits 31:30 and masked is the fp32 value 2t;
        // rv holds r/2, so each product is exactly +-r or 0
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          acc[kk] = fmaf(__uint_as_float((wv[u].x << (30 - 2 * kk)) & 0xC0000000u), rv[u], acc[kk]);
          acc[16 + kk] =
              fmaf(__uint_as_float((wv[u].y << (30 - 2 * kk)) & 0xC0000000u), rv[u], acc[16 + kk]);
        }
      }
    }
    // layout [q][kk][j] with an odd row stride Wp: the stores (consecutive j) and
    // the loads below (consecutive kk) both fall in distinct banks
#pragma unroll
    for (int u = 0; u < 32; ++u) red[(size_t)q * 32 * Wp + u * Wp + j] = acc[u];
  }
  unit_sync(cx);
  float* out = P.partial + ((size_t)ts * d.nb + b) * 2 * I;
  for (int o = cx.ut; o < 2 * I; o += cx.UT) {
    const int jj = o / 32, kk = o % 32;
    float s = 0.f;
    for (int qq = 0; qq < Q; ++qq) s += red[(size_t)qq * 32 * Wp + kk * Wp + jj];
    const int gv = jj / half;
    const int i = (jj % half) * 32 + kk;
    out[gv * I + i] = s * __half2float(alpha[gv * I + i]);
  }
  // publish: the barrier orders the unit's stores before the leader's fence + add
  unit_sync(cx);
  if (cx.ut == 0) {
    __threadfence();
    atomicAdd(P.sync + so.slot + ts, 1u);
  }
  return true;
}

// Score the channels of one (token, slot) once all its blocks are in: sum
// the block partials in block order, s = w ||d|| |phi(ghat) vhat|.
__device__ bool score_task(const Params& P, int ts, int* flag) {
  const Dims& d = P.d;
  const SyncOff so = sync_offsets(d);
  const int t = ts / d.topk, slot = ts % d.topk, I = d.I;
  if (threadIdx.x == 0)
    *flag = wait_at_least(P.sync + so.slot + ts, (uint32_t)d.nb, P.sync + kSyncAbort, P.err);
  __syncthreads();
  if (!*flag) return false;
  int e = P.ids_in[ts];
  if (e < 0 || e >= d.E) e = 0;
  const float wv = P.w_in[ts];
  for (int i = threadIdx.x; i < I; i += kThreads) {
    const float* pg = P.partial + ((size_t)ts * d.nb) * 2 * I + i;
    float g = 0.f, v = 0.f;
    int bb = 0;
    for (; bb + 16 <= d.nb; bb += 16) {   // loads first, then the sums in block order
      float gg[16], vv[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        gg[u] = __ldcg(pg + (size_t)(bb + u) * 2 * I);
        vv[u] = __ldcg(pg + (size_t)(bb + u) * 2 * I + I);
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        g += gg[u];
        v += vv[u];
      }
    }
    for (; bb < d.nb; ++bb) {
      g += __ldcg(pg + (size_t)bb * 2 * I);
      v += __ldcg(pg + (size_t)bb * 2 * I + I);
    }
    const float pv = silu_f(g) * v;
    const float s = wv * __ldg(P.dnorm + (size_t)e * I + i) * fabsf(pv);
    const size_t o = (size_t)t * d.N + (size_t)slot * I + i;
    P.ghat[o] = g;
    P.vhat[o] = v;
    P.p[o] = pv;
    P.score[o] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(P.sync + so.tok + t, 1u);
  }
  return true;
}

// ------------------------------- phase 2 -----------------------------------
__device__ __forceinline__ void dot8(const uint4& q, const float4& xa, const float4& xb, float& s) {
  s = fmaf(bf16_lo(q.x), xa.x, s); s = fmaf(bf16_hi(q.x), xa.y, s);
  s = fmaf(bf16_lo(q.y), xa.z, s); s = fmaf(bf16_hi(q.y), xa.w, s);
  s = fmaf(bf16_lo(q.z), xb.x, s); s = fmaf(bf16_hi(q.z), xb.y, s);
  s = fmaf(bf16_lo(q.w), xb.z, s); s = fmaf(bf16_hi(q.w), xb.w, s);
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p));
}

__device__ void kept_item(const Params& P, int t, int qi, int lane) {
  const Dims& d = P.d;
  const int n = __ldcg(P.kept + (size_t)t * d.N + qi);
  const int slot = n / d.I, i = n % d.I;
  const int e = __ldcg(P.ids_ws + t * d.topk + slot);
  const size_t row = (size_t)e * d.I + i;
  // the output phase reads this channel's transposed down row in 32-byte
  // pieces from many CTAs: bring the whole row into L2 now
  {
    const char* dt = reinterpret_cast<const char*>(P.Dt + row * d.H);
    for (int off = lane * 128; off < d.H * 2; off += 32 * 128) prefetch_l2(dt + off);
  }
  const uint4* g4 = reinterpret_cast<const uint4*>(P.G + row * d.H);
  const uint4* v4 = reinterpret_cast<const uint4*>(P.V + row * d.H);
  const float4* x4 = reinterpret_cast<const float4*>(P.x + (size_t)t * d.H);
  float sg = 0.f, sv = 0.f;
  const int n8 = d.H / 8;
  int h8 = lane;
  constexpr int kU = 8;   // 16-byte loads per lane and row issued together
  for (; h8 + 32 * (kU - 1) < n8; h8 += 32 * kU) {
    uint4 gq[kU], vq[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      gq[u] = ldg_nc4(g4 + h8 + 32 * u);
      vq[u] = ldg_nc4(v4 + h8 + 32 * u);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const float4 xa = __ldg(x4 + 2 * (h8 + 32 * u)), xb = __ldg(x4 + 2 * (h8 + 32 * u) + 1);
      dot8(gq[u], xa, xb, sg);
      dot8(vq[u], xa, xb, sv);
    }
  }
  for (; h8 < n8; h8 += 32) {
    const uint4 gq = ldg_nc4(g4 + h8), vq = ldg_nc4(v4 + h8);
    const float4 xa = __ldg(x4 + 2 * h8), xb = __ldg(x4 + 2 * h8 + 1);
    dot8(gq, xa, xb, sg);
    dot8(vq, xa, xb, sv);
  }
  sg = warp_sum(sg);
  sv = warp_sum(sv);
  if (lane == 0) {
    P.wa[(size_t)t * d.N + qi] = __ldcg(P.w_ws + t * d.topk + slot) * silu_f(sg) * sv;
    P.rowoff[(size_t)t * d.N + qi] = (int32_t)row;
  }
}

__device__ void recovery_item(const Params& P, int t, int ch, int lane) {
  // 64 channels: lane l takes channels l and l + 32 (full b rows), then the
  // warp transposes and sums the 32 lane vectors; lane j ends with component j
  const Dims& d = P.d;
  const int n0 = ch * 64;
  const int slot = n0 / d.I;
  const int e = __ldcg(P.ids_ws + t * d.topk + slot);
  const float wv = __ldcg(P.w_ws + t * d.topk + slot);
  const uint32_t kb0 = __ldcg(P.keptbits + (size_t)t * (d.N / 32) + ch * 2);
  const uint32_t kb1 = __ldcg(P.keptbits + (size_t)t * (d.N / 32) + ch * 2 + 1);
  const bool s0 = !((kb0 >> lane) & 1u), s1 = !((kb1 >> lane) & 1u);
  const float c0 = s0 ? wv * __ldcg(P.p + (size_t)t * d.N + n0 + lane) : 0.f;
  const float c1 = s1 ? wv * __ldcg(P.p + (size_t)t * d.N + n0 + 32 + lane) : 0.f;
  const __half* b0 = P.bco + ((size_t)e * d.I + (n0 % d.I) + lane) * d.r;
  const __half* b1 = b0 + (size_t)32 * d.r;
  for (int j0 = 0; j0 < d.r; j0 += 32) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = 0.f;
    const int jn = min(32, d.r - j0);
    if ((d.r & 7) == 0) {
      // rows are 16-byte aligned: 8 components per load
      uint4 q0[4], q1[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool in = 8 * u < jn;
        q0[u] = (in && s0) ? ldg_nc4(b0 + j0 + 8 * u) : make_uint4(0, 0, 0, 0);
        q1[u] = (in && s1) ? ldg_nc4(b1 + j0 + 8 * u) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t w0[4] = {q0[u].x, q0[u].y, q0[u].z, q0[u].w};
        const uint32_t w1[4] = {q1[u].x, q1[u].y, q1[u].z, q1[u].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&w0[h]));
          const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&w1[h]));
          v[8 * u + 2 * h] = fmaf(c1, f1.x, c0 * f0.x);
          v[8 * u + 2 * h + 1] = fmaf(c1, f1.y, c0 * f0.y);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (j < jn) {
          const float x0 = s0 ? c0 * __half2float(b0[j0 + j]) : 0.f;
          v[j] = s1 ? fmaf(c1, __half2float(b1[j0 + j]), x0) : x0;
        }
      }
    }
    // recursive halving: after 5 rounds lane l holds the warp sum of component l
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int j = 0; j < off; ++j) {
        const float send = upper ? v[j] : v[j + off];
        const float keep = upper ? v[j + off] : v[j];
        v[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
    if (lane < jn) atomicAdd(P.cvec + (size_t)t * d.r + j0 + lane, v[0]);
  }
}

// ------------------------------- phase 3 -----------------------------------
__device__ __forceinline__ void axpy8(float c, const uint4& v, float* acc) {
  acc[0] = fmaf(c, bf16_lo(v.x), acc[0]); acc[1] = fmaf(c, bf16_hi(v.x), acc[1]);
  acc[2] = fmaf(c, bf16_lo(v.y), acc[2]); acc[3] = fmaf(c, bf16_hi(v.y), acc[3]);
  acc[4] = fmaf(c, bf16_lo(v.z), acc[4]); acc[5] = fmaf(c, bf16_hi(v.z), acc[5]);
  acc[6] = fmaf(c, bf16_lo(v.w), acc[6]); acc[7] = fmaf(c, bf16_hi(v.w), acc[7]);
}

constexpr int kTokGroup = 2;
constexpr int kRowBatch = 4;   // rows per token and thread whose loads are issued together

// One output item: 16 columns h0..h0+15 (one 32-byte piece of every kept
// transposed down row) for tokens t0, t0+1.  Thread (rg, half): rows
// rg, rg+256, ...; 8 columns each.  y = sum_K (w a)_j Dt_j + U c.
__device__ void out_item(const Params& P, int s, int t0, unsigned char* smem) {
  const Dims& d = P.d;
  float* wred = reinterpret_cast<float*>(smem);        // [kTokGroup][kWarps][16]
  float* us = wred + kTokGroup * kWarps * 16;          // [16][r]  U rows of the slice
  float* cs = us + 16 * kMaxRank;                      // [kTokGroup][r] recovery vectors
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int h0 = s * 16;
  const bool recover = P.k < d.N;
  if (recover) {
    for (int q = threadIdx.x; q < 16 * d.r; q += kThreads) {
      const int h = h0 + q / d.r;
      us[q] = h < d.H ? __half2float(P.U[(size_t)h * d.r + q % d.r]) : 0.f;
    }
    for (int q = threadIdx.x; q < kTokGroup * d.r; q += kThreads) {
      const int t = t0 + q / d.r;
      cs[q] = t < P.B ? __ldcg(P.cvec + (size_t)t * d.r + q % d.r) : 0.f;
    }
  }
  const int rg = threadIdx.x >> 1, hf = threadIdx.x & 1;   // 256 row groups x 2 halves
  const int hh = h0 + hf * 8;
  float acc[kTokGroup][8];
#pragma unroll
  for (int tt = 0; tt < kTokGroup; ++tt)
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[tt][u] = 0.f;
  if (hh < d.H) {
    for (int q0 = rg; q0 < P.k; q0 += 256 * kRowBatch) {
      int32_t r[kTokGroup][kRowBatch];
      float c[kTokGroup][kRowBatch];
#pragma unroll
      for (int tt = 0; tt < kTokGroup; ++tt)
#pragma unroll
        for (int u = 0; u < kRowBatch; ++u) {
          const int q = q0 + 256 * u;
          const bool ok = t0 + tt < P.B && q < P.k;
          r[tt][u] = ok ? __ldcg(P.rowoff + (size_t)(t0 + tt) * d.N + q) : -1;
          c[tt][u] = ok ? __ldcg(P.wa + (size_t)(t0 + tt) * d.N + q) : 0.f;
        }
      uint4 v[kTokGroup][kRowBatch];
#pragma unroll
      for (int tt = 0; tt < kTokGroup; ++tt)
#pragma unroll
        for (int u = 0; u < kRowBatch; ++u)
          v[tt][u] = r[tt][u] >= 0 ? __ldcg(reinterpret_cast<const uint4*>(P.Dt + (size_t)r[tt][u] * d.H + hh))
                                   : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int tt = 0; tt < kTokGroup; ++tt)
#pragma unroll
        for (int u = 0; u < kRowBatch; ++u) axpy8(c[tt][u], v[tt][u], acc[tt]);
    }
  }
  // sum the 16 row groups of the warp (lane bits 1..4), then the 16 warps
#pragma unroll
  for (int tt = 0; tt < kTokGroup; ++tt)
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int o = 2; o < 32; o <<= 1) acc[tt][u] += __shfl_xor_sync(0xffffffffu, acc[tt][u], o);
  if (lane < 2)
#pragma unroll
    for (int tt = 0; tt < kTokGroup; ++tt)
#pragma unroll
      for (int u = 0; u < 8; ++u) wred[(tt * kWarps + warp) * 16 + lane * 8 + u] = acc[tt][u];
  __syncthreads();
  if (threadIdx.x < 16 * kTokGroup) {
    const int tt = threadIdx.x >> 4, col = threadIdx.x & 15;
    const int t = t0 + tt, h = h0 + col;
    if (t < P.B && h < d.H) {
      float sum = 0.f;
      for (int w = 0; w < kWarps; ++w) sum += wred[(tt * kWarps + w) * 16 + col];
      if (recover)
        for (int jj = 0; jj < d.r; ++jj) sum = fmaf(us[col * d.r + jj], cs[tt * d.r + jj], sum);
      P.y[(size_t)t * d.H + h] = sum;
    }
  }
  __syncthreads();
}

// ------------------------------- the kernel --------------------------------
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const Params P) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int ctl[2];
  if (threadIdx.x == 0) ctl[0] = 0;
  const Dims& d = P.d;
  const SyncOff so = sync_offsets(d);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nctas = gridDim.x;
  uint32_t* abort_flag = P.sync + kSyncAbort;
  unsigned long long* stamp = P.stamps ? P.stamps + (size_t)blockIdx.x * 5 : nullptr;
  if (stamp && threadIdx.x == 0) stamp[0] = globaltimer();

  // phase 0: rotations, one warp per (token, block), spread over CTAs first
  {
    const int items = P.B * d.nb;
    for (int it = blockIdx.x + nctas * warp; it < items; it += nctas * kWarps)
      rotate_item(P, it / d.nb, it % d.nb, lane);
  }
  if (stamp) {
    __syncthreads();
    if (threadIdx.x == 0) stamp[1] = globaltimer();
  }
  // phase 1a: screen units (token, slot, block) from a shared queue
  {
    const int units = P.B * d.topk * d.nb;
    const bool halves = units > nctas;
    const int UT = halves ? kThreads / 2 : kThreads;
    const int hid = halves ? (int)(threadIdx.x / UT) : 0;
    UnitCtx cx;
    cx.ut = threadIdx.x - hid * UT;
    cx.UT = UT;
    cx.bar = 1 + hid;
    cx.sm = smem + (size_t)hid * unit_smem_bytes(d.I, unit_groups(P.W8, UT));
    int* next = reinterpret_cast<int*>(cx.sm + 4 * (size_t)d.I + kBlock * 8);   // flags[0..3]
    if (cx.ut == 0) next[1] = (int)atomicAdd(P.sync + kSyncNext, 1u);
    unit_sync(cx);
    int u = next[1];
    bool ok = true;
    while (u < units) {
      // take the following unit now so the round trip overlaps this one
      if (cx.ut == 0) next[2] = (int)atomicAdd(P.sync + kSyncNext, 1u);
      const int b = u % d.nb, ts = u / d.nb;
      if (!screen_unit(P, ts / d.topk, ts % d.topk, b, cx)) {
        ok = false;
        break;
      }
      unit_sync(cx);
      u = next[2];
      unit_sync(cx);
    }
    if (!ok) ctl[0] = 1;
    __syncthreads();
    if (ctl[0] == 1) return;
  }
  // phase 1b: scoring tasks, then 1c: top-k tasks, spread over the CTAs
  {
    int* flag = reinterpret_cast<int*>(smem);
    for (int ts = blockIdx.x; ts < P.B * d.topk; ts += nctas) {
      if (!score_task(P, ts, flag)) return;
      __syncthreads();
    }
    for (int t = blockIdx.x; t < P.B; t += nctas) {
      if (threadIdx.x == 0)
        ctl[1] = wait_at_least(P.sync + so.tok + t, (uint32_t)d.topk, abort_flag, P.err);
      __syncthreads();
      if (!ctl[1]) return;
      topk_token(P, t, smem);
      __syncthreads();
    }
  }
  if (stamp && threadIdx.x == 0) stamp[2] = globaltimer();
  // phase 2: kept channels and recovery chunks, one warp each
  const int per_tok = P.k + d.N / 64;
  const long long M = (long long)P.B * per_tok;
  {
    const long long wtot = (long long)nctas * kWarps;
    const long long gw = (long long)blockIdx.x * kWarps + warp;
    int cur_t = -1;
    for (long long q = gw; q < M; q += wtot) {
      const int t = (int)(q / per_tok), local = (int)(q % per_tok);
      if (t != cur_t) {
        int w_ok = 1;
        if (lane == 0) w_ok = wait_at_least(P.sync + so.flag + t, 1u, abort_flag, P.err);
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) break;
        __syncwarp();
        cur_t = t;
      }
      if (local < P.k)
        kept_item(P, t, local, lane);
      else
        recovery_item(P, t, local - P.k, lane);
    }
  }
  __syncthreads();
  if (stamp && threadIdx.x == 0) stamp[3] = globaltimer();
  if (threadIdx.x == 0) {
    __threadfence();
    int ok = ld_acquire(abort_flag) == 0u;
    if (ok) {
      long long mine = 0;
      const long long wtot = (long long)nctas * kWarps;
      for (int w = 0; w < kWarps; ++w) {
        const long long gw = (long long)blockIdx.x * kWarps + w;
        if (gw < M) mine += (M - 1 - gw) / wtot + 1;
      }
      atomicAdd(P.sync + kSyncExact, (uint32_t)mine);
      ok = wait_at_least(P.sync + kSyncExact, (uint32_t)M, abort_flag, P.err);
    }
    ctl[1] = ok;
  }
  __syncthreads();
  if (!ctl[1]) return;
  // phase 3: output items (16-column slice, token pair)
  {
    const int slices = (d.H + 15) / 16;
    const int groups = (P.B + kTokGroup - 1) / kTokGroup;
    for (int it = blockIdx.x; it < slices * groups; it += nctas)
      out_item(P, it % slices, (it / slices) * kTokGroup, smem);
  }
  if (stamp && threadIdx.x == 0) stamp[4] = globaltimer();
  // the last CTA out resets the synchronisation area for the next call
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    ctl[0] = atomicAdd(P.sync + kSyncDone, 1u) == (uint32_t)(nctas - 1);
  }
  __syncthreads();
  if (ctl[0]) {
    for (int i = threadIdx.x; i < P.B * d.nb; i += kThreads) P.sync[so.rot + i] = 0u;
    for (int i = threadIdx.x; i < P.B * d.topk; i += kThreads) P.sync[so.slot + i] = 0u;
    for (int i = threadIdx.x; i < P.B; i += kThreads) {
      P.sync[so.tok + i] = 0u;
      P.sync[so.flag + i] = 0u;
    }
    if (threadIdx.x == 0) {
      P.sync[kSyncExact] = 0u;
      P.sync[kSyncNext] = 0u;
      P.sync[kSyncDone] = 0u;
    }
  }
}

int screen_groups(const Dims& d) {
  const int W8 = d.I / 16;
  int Q = kThreads / W8;
  if (Q > kMaxGroups) Q = kMaxGroups;
  if (Q < 1) Q = 1;
  return Q;
}

size_t decode_smem_bytes(const Dims& d) {
  const size_t whole = unit_smem_bytes(d.I, unit_groups(d.I / 16, kThreads));
  const size_t halves = 2 * unit_smem_bytes(d.I, unit_groups(d.I / 16, kThreads / 2));
  const size_t screen = whole > halves ? whole : halves;
  const size_t topk = topk_smem_bytes(d.N);
  const size_t out = ((size_t)kTokGroup * kWarps * 16 + 16 * kMaxRank + kTokGroup * kMaxRank) * 4;
  const size_t m = screen > topk ? screen : topk;
  return m > out ? m : out;
}

}  // namespace

size_t sync_words(const Dims& d) { return (size_t)sync_offsets(d).total; }

cudaError_t configure_decode_kernels(const Dims& d) {
  const size_t smem = decode_smem_bytes(d);
  cudaFuncAttributes fa;
  cudaError_t err = cudaFuncGetAttributes(&fa, decode_kernel);
  if (err != cudaSuccess) return err;
  if ((size_t)fa.maxDynamicSharedSizeBytes < smem)
    err = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
  return err;
}

int decode_grid(const Dims& d) {
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel, kThreads,
                                                    decode_smem_bytes(d)) != cudaSuccess)
    return 0;
  return per_sm >= 1 ? sms : 0;   // one CTA per SM, all co-resident
}

cudaError_t launch_decode(const moe_reader& h, const float* x, int B, const int32_t* ids,
                          const float* w, int k, float* y, cudaStream_t s, const cudaEvent_t* ev,
                          unsigned long long* stamps) {
  const Dims& d = h.d;
  const Workspace& ws = h.ws;
  cudaError_t err;
  unsigned int rec_flags = cudaEventRecordDefault;
  if (ev) {
    // inside stream capture a plain record is only a dependency marker; the
    // External flag makes it an event-record node of the graph
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if ((err = cudaStreamIsCapturing(s, &cs)) != cudaSuccess) return err;
    if (cs == cudaStreamCaptureStatusActive) rec_flags = cudaEventRecordExternal;
    if ((err = cudaEventRecordWithFlags(ev[0], s, rec_flags)) != cudaSuccess) return err;
  }
  Params P;
  P.d = d;
  P.B = B;
  P.k = k;
  P.x = x;
  P.ids_in = ids;
  P.w_in = w;
  P.y = y;
  P.sigma = h.p.sigma;
  P.codes = h.p.codes;
  P.scales = h.p.scales;
  P.dnorm = h.p.dnorm;
  P.G = h.G;
  P.V = h.V;
  P.Dt = h.p.Dt;
  P.U = h.p.U;
  P.bco = h.p.b;
  P.ids_ws = ws.ids;
  P.w_ws = ws.w;
  P.rx = ws.rx;
  P.mask = ws.mask;
  P.partial = ws.partial;
  P.ghat = ws.ghat;
  P.vhat = ws.vhat;
  P.p = ws.p;
  P.score = ws.score;
  P.keptbits = ws.keptbits;
  P.kept = ws.kept;
  P.rowoff = ws.rowoff;
  P.wa = ws.wa;
  P.cvec = ws.cpart;
  P.stamps = stamps;
  P.sync = ws.sync;
  P.err = ws.err;
  P.Q = screen_groups(d);
  P.W8 = d.I / 16;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(h.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = decode_smem_bytes(d);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if ((err = cudaLaunchKernelEx(&cfg, decode_kernel, P)) != cudaSuccess) return err;
  if (ev && (err = cudaEventRecordWithFlags(ev[1], s, rec_flags)) != cudaSuccess) return err;
  return cudaSuccess;
}

}  // namespace mr
