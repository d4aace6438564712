// C ABI of the channel reader: argument checks, device memory ownership and
// the order of launches.  Every computational step runs in the kernels of
// prepare_sketch.cu, prepare_svd.cu and decode.cu.
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <vector>

#include "internal.cuh"

namespace {

// Pending one-shot fault injections that are not tied to a handle.
std::atomic<int> g_fail_next_alloc{0};
std::atomic<int> g_stall_next_prepare{0};

using mr::Dims;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_config(const moe_reader_config* c) {
  if (!c) return MOE_READER_EINVAL;
  if (c->flags & ~(MOE_READER_FLAG_RHO_RANK | MOE_READER_FLAG_TRIT5)) return MOE_READER_EINVAL;
  if ((c->flags & MOE_READER_FLAG_RHO_RANK) && c->screen_coords != mr::kBlock)
    return MOE_READER_EINVAL;   // the expected-error ranking reads the whole sketch
  if (c->hidden < 8 || c->hidden % 8 != 0 || c->hidden > 65536) return MOE_READER_EINVAL;
  if (c->num_experts < 1 || c->num_experts > 65536) return MOE_READER_EINVAL;
  if (c->experts_per_token < 1 || c->experts_per_token > std::min(c->num_experts, mr::kMaxTopk))
    return MOE_READER_EINVAL;
  if (c->inter < 64 || c->inter % 64 != 0 || c->inter > mr::kMaxInter) return MOE_READER_EINVAL;
  if ((long long)c->experts_per_token * c->inter > 32768) return MOE_READER_EINVAL;
  if ((long long)c->num_experts * c->inter >= (1LL << 30)) return MOE_READER_EINVAL;
  if (c->screen_coords < 1 || c->screen_coords > mr::kBlock) return MOE_READER_EINVAL;
  if (c->rank < 1 || c->rank > std::min(c->hidden, mr::kMaxRank)) return MOE_READER_EINVAL;
  if (c->max_batch < 1 || c->max_batch > mr::kMaxBatch) return MOE_READER_EINVAL;
  return MOE_READER_OK;
}

Dims make_dims(const moe_reader_config& c) {
  Dims d;
  d.H = c.hidden;
  d.E = c.num_experts;
  d.topk = c.experts_per_token;
  d.I = c.inter;
  d.c = c.screen_coords;
  d.r = c.rank;
  d.Bmax = c.max_batch;
  d.nb = (d.H + mr::kBlock - 1) / mr::kBlock;
  d.Hp = d.nb * mr::kBlock;
  d.N = d.topk * d.I;
  d.trit5 = (c.flags & MOE_READER_FLAG_TRIT5) ? 1 : 0;
  const int run2 = (d.I + 3) / 4, run5 = (d.I + 4) / 5;
  d.S2b = ((run2 + mr::kSector - 1) / mr::kSector) * mr::kSector;
  d.S = d.trit5 ? ((run5 + mr::kSector - 1) / mr::kSector) * mr::kSector : d.S2b;
  d.runW = d.trit5 ? (run5 + 3) / 4 : d.I / 16;
  d.rho_rank = (c.flags & MOE_READER_FLAG_RHO_RANK) ? 1 : 0;
  return d;
}

// A bump allocator over one cudaMalloc: every sub-array starts on 256 bytes.
struct Arena {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) & ~(size_t)255;
    return o;
  }
};

struct Allocs {
  void* prepared = nullptr;
  void* workspace = nullptr;
};

void free_handle_memory(moe_reader* h) {
  if (!h) return;
  if (h->p.codes) cudaFree(h->p.codes);   // start of the prepared block
  if (h->ws.mask) cudaFree(h->ws.mask);   // start of the workspace block
  h->p.codes = nullptr;
  h->ws.mask = nullptr;
}

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_READER_OK;
  if (e == cudaErrorMemoryAllocation) return MOE_READER_ENOMEM;
  return MOE_READER_ECUDA;
}

int64_t export_size(const moe_reader* h, int which) {
  const Dims& d = h->d;
  const int64_t B = h->has_decode ? h->last_B : -1;
  switch (which) {
    case MOE_READER_EXPORT_CODES: return (int64_t)d.E * d.nb * mr::kBlock * 2 * d.S;
    case MOE_READER_EXPORT_SCALES:
    case MOE_READER_EXPORT_RHO: return (int64_t)d.E * d.nb * 2 * d.I * 2;
    case MOE_READER_EXPORT_DNORM: return (int64_t)d.E * d.I * 4;
    case MOE_READER_EXPORT_DT: return (int64_t)d.E * d.I * d.H * 2;
    case MOE_READER_EXPORT_U: return (int64_t)d.H * d.r * 2;
    case MOE_READER_EXPORT_B: return (int64_t)d.E * d.I * d.r * 2;
    case MOE_READER_EXPORT_SIGMA: return (int64_t)d.Hp;
    case MOE_READER_EXPORT_EIGVALS: return (int64_t)d.r * 8;
    case MOE_READER_EXPORT_MASK: return B < 0 ? MOE_READER_ESTATE : B * d.nb * 4 * 4;
    case MOE_READER_EXPORT_GHAT:
    case MOE_READER_EXPORT_VHAT:
    case MOE_READER_EXPORT_SCORE: return B < 0 ? MOE_READER_ESTATE : B * d.N * 4;
    default: return MOE_READER_EINVAL;
  }
}

const void* export_ptr(const moe_reader* h, int which) {
  switch (which) {
    case MOE_READER_EXPORT_CODES: return h->p.codes;
    case MOE_READER_EXPORT_SCALES: return h->p.scales;
    case MOE_READER_EXPORT_RHO: return h->p.rho;
    case MOE_READER_EXPORT_DNORM: return h->p.dnorm;
    case MOE_READER_EXPORT_DT: return h->p.Dt;
    case MOE_READER_EXPORT_U: return h->p.U;
    case MOE_READER_EXPORT_B: return h->p.b;
    case MOE_READER_EXPORT_SIGMA: return h->p.sigma;
    case MOE_READER_EXPORT_EIGVALS: return h->p.eigvals;
    case MOE_READER_EXPORT_MASK: return h->ws.mask;
    case MOE_READER_EXPORT_GHAT: return h->ws.ghat;
    case MOE_READER_EXPORT_VHAT: return h->ws.vhat;
    case MOE_READER_EXPORT_SCORE: return h->ws.score;
    default: return nullptr;
  }
}

int check_decode_args(const moe_reader* h, const void* x, int32_t B, const void* ids,
                      const void* w, int32_t k, const void* y) {
  if (!h) return MOE_READER_EINVAL;
  if (B < 0 || B > h->d.Bmax) return MOE_READER_EINVAL;
  if (k < 0 || k > h->d.N) return MOE_READER_EINVAL;
  if (B == 0) return MOE_READER_OK;
  if (!x || !ids || !w || !y) return MOE_READER_EINVAL;
  return MOE_READER_OK;
}

// Next profiling slot (events + stamp rows), or -1 when profiling is off.
// Slots wrap after kProfSlots decode calls.
int profile_slot(moe_reader* h) {
  if (!h->prof_on) return -1;
  const int slot = h->prof_used % mr::kProfSlots;
  h->prof_used++;
  return slot;
}

cudaError_t launch_profiled(moe_reader* h, const float* x, int B, const int32_t* ids,
                            const float* w, int k, float* y, cudaStream_t s, bool shared = false) {
  const int slot = profile_slot(h);
  if (slot < 0) return mr::launch_decode(*h, x, B, ids, w, k, y, s, nullptr, nullptr, shared);
  return mr::launch_decode(*h, x, B, ids, w, k, y, s, h->prof_ev[slot],
                           h->prof_stamps + (size_t)slot * h->grid * 5, shared);
}

}  // namespace

namespace mr {

cudaError_t device_alloc(void** p, size_t bytes) {
  *p = nullptr;
  if (g_fail_next_alloc.exchange(0)) return cudaErrorMemoryAllocation;
  return cudaMalloc(p, bytes);
}

bool take_prepare_stall() { return g_stall_next_prepare.exchange(0) != 0; }

}  // namespace mr

extern "C" {

int moe_reader_abi_version(void) { return MOE_READER_ABI_VERSION; }

const char* moe_reader_strerror(int code) {
  switch (code) {
    case MOE_READER_OK: return "ok";
    case MOE_READER_EINVAL: return "invalid argument (config, shape, k, batch, pointer or alignment)";
    case MOE_READER_ENOMEM: return "device allocation failed";
    case MOE_READER_ECUDA: return "CUDA runtime call failed";
    case MOE_READER_ETIMEOUT: return "a bounded device wait timed out";
    case MOE_READER_EDEVICE: return "device-side input check failed (expert ids, weights or x)";
    case MOE_READER_ESTATE: return "no completed decode on this handle";
    case MOE_READER_ETOOBIG:
      return "rows*cols exceeds the 2^18-element fixed scratch of moe_reader_topk_noalloc";
    default: return "unknown status";
  }
}

int moe_reader_prepare(const moe_reader_config* cfg, const void* gate, const void* up,
                       const void* down, const int8_t* sigma, void* stream, moe_reader_t** out) {
  if (!out) return MOE_READER_EINVAL;
  *out = nullptr;
  int st = check_config(cfg);
  if (st != MOE_READER_OK) return st;
  if (!gate || !up || !down || !sigma) return MOE_READER_EINVAL;
  if (!aligned(gate, 256) || !aligned(up, 256) || !aligned(down, 256)) return MOE_READER_EINVAL;
  const Dims d = make_dims(*cfg);
  for (int i = 0; i < d.Hp; ++i)
    if (sigma[i] != 1 && sigma[i] != -1) return MOE_READER_EINVAL;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  moe_reader* h = static_cast<moe_reader*>(calloc(1, sizeof(moe_reader)));
  if (!h) return MOE_READER_ENOMEM;
  h->cfg = *cfg;
  h->d = d;
  cudaGetDevice(&h->device);
  h->G = static_cast<const __nv_bfloat16*>(gate);
  h->V = static_cast<const __nv_bfloat16*>(up);

  // ---- prepared arrays: one allocation, 256-byte aligned sub-arrays ----
  Arena pa;
  const size_t o_codes = pa.take((size_t)d.E * d.nb * mr::kBlock * 2 * d.S);
  const size_t o_scales = pa.take((size_t)d.E * d.nb * 2 * d.I * 2);
  const size_t o_rho = pa.take((size_t)d.E * d.nb * 2 * d.I * 2);
  const size_t o_dnorm = pa.take((size_t)d.E * d.I * 4);
  const size_t o_dt = pa.take((size_t)d.E * d.I * d.H * 2);
  const size_t o_u = pa.take((size_t)d.H * d.r * 2);
  const size_t o_ut = pa.take((size_t)d.H * d.r * 2);
  const size_t o_b = pa.take((size_t)d.E * d.I * d.r * 2);
  const size_t o_sigma = pa.take((size_t)d.Hp);
  const size_t o_eig = pa.take((size_t)d.r * 8);
  const size_t o_bn2 = pa.take((size_t)d.E * d.I * 4);
  void* pbase = nullptr;
  cudaError_t ce = mr::device_alloc(&pbase, pa.off);
  if (ce != cudaSuccess) {
    free(h);
    return cuda_status(ce);
  }
  char* pb = static_cast<char*>(pbase);
  h->p.codes = reinterpret_cast<uint8_t*>(pb + o_codes);
  h->p.scales = reinterpret_cast<__half*>(pb + o_scales);
  h->p.rho = reinterpret_cast<__half*>(pb + o_rho);
  h->p.dnorm = reinterpret_cast<float*>(pb + o_dnorm);
  h->p.bnorm2 = reinterpret_cast<float*>(pb + o_bn2);
  h->p.Dt = reinterpret_cast<__nv_bfloat16*>(pb + o_dt);
  h->p.U = reinterpret_cast<__half*>(pb + o_u);
  h->p.Ut = reinterpret_cast<__half*>(pb + o_ut);
  h->p.b = reinterpret_cast<__half*>(pb + o_b);
  h->p.sigma = reinterpret_cast<int8_t*>(pb + o_sigma);
  h->p.eigvals = reinterpret_cast<double*>(pb + o_eig);
  h->resident[0] = o_scales - o_codes;
  h->resident[1] = o_rho - o_scales;
  h->resident[2] = o_dnorm - o_rho;
  h->resident[3] = o_dt - o_dnorm;
  h->resident[4] = o_u - o_dt;
  h->resident[5] = o_b - o_u;
  h->resident[6] = o_sigma - o_b;
  h->resident[7] = o_eig - o_sigma;

  // ---- decode workspace ----
  const size_t Bm = (size_t)d.Bmax;
  Arena wa;
  const size_t w_mask = wa.take(Bm * d.nb * 16);
  const size_t w_ids = wa.take(Bm * d.topk * 4);
  const size_t w_w = wa.take(Bm * d.topk * 4);
  const size_t w_part = wa.take(Bm * d.topk * d.nb * 2 * d.I * 4);
  const size_t w_ghat = wa.take(Bm * d.N * 4);
  const size_t w_vhat = wa.take(Bm * d.N * 4);
  const size_t w_p = wa.take(Bm * d.N * 4);
  const size_t w_score = wa.take(Bm * d.N * 4);
  const size_t w_kb = wa.take(Bm * (d.N / 32) * 4);
  const size_t w_kept = wa.take(Bm * d.N * 4);
  const size_t w_wa = wa.take(Bm * d.N * 4);
  const size_t w_sync = wa.take(mr::sync_words(d) * 4);
  const size_t w_cp = wa.take(Bm * d.r * 4);
  const size_t w_xs = wa.take(Bm * d.H * 4);
  const size_t w_ys = wa.take(Bm * d.H * 4);
  const size_t w_hs = wa.take(Bm * d.H * 4);
  const size_t w_xsc = wa.take(Bm * 4);
  const size_t w_rn2 = wa.take(Bm * d.nb * 4);
  const size_t EI = (size_t)d.E * d.I;
  const size_t w_ssc = wa.take(EI * 4);
  const size_t w_skp = wa.take(EI * 4);
  const size_t w_sbt = wa.take(EI / 32 * 4);
  const size_t w_est = wa.take(((size_t)d.E + 1) * 4);
  const size_t w_els = wa.take(Bm * d.topk * 4);
  const size_t w_kct = wa.take(Bm * 4);
  const size_t w_sK = wa.take(4);
  const size_t w_sinf = wa.take(EI * 4);
  const size_t w_is = wa.take(Bm * d.topk * 4);
  const size_t w_ws = wa.take(Bm * d.topk * 4);
  const size_t w_bmc = wa.take((size_t)d.E * d.nb * 16);
  const size_t w_bmk = wa.take((size_t)d.E * (d.I / 32) * 4);
  const size_t w_bms = wa.take((size_t)d.E * (d.I / 32) * 4);
  const size_t w_bme = wa.take((size_t)((d.E + 31) / 32) * 4);
  const size_t w_cnt = wa.take(16 * 8);
  const size_t w_err = wa.take(4);
  void* wbase = nullptr;
  ce = mr::device_alloc(&wbase, wa.off);
  if (ce != cudaSuccess) {
    cudaFree(pbase);
    free(h);
    return cuda_status(ce);
  }
  char* wb = static_cast<char*>(wbase);
  h->ws.mask = reinterpret_cast<uint32_t*>(wb + w_mask);
  h->ws.ids = reinterpret_cast<int32_t*>(wb + w_ids);
  h->ws.w = reinterpret_cast<float*>(wb + w_w);
  h->ws.partial = reinterpret_cast<float*>(wb + w_part);
  h->ws.ghat = reinterpret_cast<float*>(wb + w_ghat);
  h->ws.vhat = reinterpret_cast<float*>(wb + w_vhat);
  h->ws.p = reinterpret_cast<float*>(wb + w_p);
  h->ws.score = reinterpret_cast<float*>(wb + w_score);
  h->ws.keptbits = reinterpret_cast<uint32_t*>(wb + w_kb);
  h->ws.kept = reinterpret_cast<int32_t*>(wb + w_kept);
  h->ws.wa = reinterpret_cast<float*>(wb + w_wa);
  h->ws.sync = reinterpret_cast<uint32_t*>(wb + w_sync);
  h->ws.cpart = reinterpret_cast<float*>(wb + w_cp);
  h->ws.x_stage = reinterpret_cast<float*>(wb + w_xs);
  h->ws.y_stage = reinterpret_cast<float*>(wb + w_ys);
  h->ws.h_stage = reinterpret_cast<float*>(wb + w_hs);
  h->ws.xscale = reinterpret_cast<float*>(wb + w_xsc);
  h->ws.rn2 = reinterpret_cast<float*>(wb + w_rn2);
  h->ws.sscore = reinterpret_cast<float*>(wb + w_ssc);
  h->ws.skept = reinterpret_cast<int32_t*>(wb + w_skp);
  h->ws.sbits = reinterpret_cast<uint32_t*>(wb + w_sbt);
  h->ws.estart = reinterpret_cast<int32_t*>(wb + w_est);
  h->ws.elist = reinterpret_cast<int32_t*>(wb + w_els);
  h->ws.kcount = reinterpret_cast<int32_t*>(wb + w_kct);
  h->ws.sK = reinterpret_cast<int32_t*>(wb + w_sK);
  h->ws.sinfo = reinterpret_cast<int32_t*>(wb + w_sinf);
  h->ws.ids_stage = reinterpret_cast<int32_t*>(wb + w_is);
  h->ws.w_stage = reinterpret_cast<float*>(wb + w_ws);
  h->ws.bm_codes = reinterpret_cast<uint32_t*>(wb + w_bmc);
  h->ws.bm_kept = reinterpret_cast<uint32_t*>(wb + w_bmk);
  h->ws.bm_skip = reinterpret_cast<uint32_t*>(wb + w_bms);
  h->ws.bm_expert = reinterpret_cast<uint32_t*>(wb + w_bme);
  h->ws.counters = reinterpret_cast<unsigned long long*>(wb + w_cnt);
  h->ws.err = reinterpret_cast<uint32_t*>(wb + w_err);
  h->resident[8] = wa.off;

  // ---- build ----
  do {
    if ((ce = cudaMemsetAsync(wbase, 0, wa.off, s)) != cudaSuccess) break;
    if ((ce = cudaMemcpyAsync(h->p.sigma, sigma, (size_t)d.Hp, cudaMemcpyHostToDevice, s)) !=
        cudaSuccess)
      break;
    if (!d.trit5) {
      if ((ce = mr::launch_sketch(d, h->G, h->V, h->p.sigma, h->p.codes, h->p.scales, h->p.rho,
                                  s)) != cudaSuccess)
        break;
    } else {
      // 2-bit runs into a scratch array, then five trits per byte into the codes
      mr::Dims d2 = d;
      d2.S = d.S2b;
      void* c2 = nullptr;
      if ((ce = mr::device_alloc(&c2, (size_t)d.E * d.nb * mr::kBlock * 2 * d.S2b)) != cudaSuccess)
        break;
      ce = mr::launch_sketch(d2, h->G, h->V, h->p.sigma, static_cast<uint8_t*>(c2), h->p.scales,
                             h->p.rho, s);
      if (ce == cudaSuccess) ce = mr::launch_pack_trit5(d, static_cast<uint8_t*>(c2), h->p.codes, s);
      if (ce == cudaSuccess) ce = cudaStreamSynchronize(s);
      cudaFree(c2);
      if (ce != cudaSuccess) break;
    }
    if ((ce = mr::launch_transpose_down(d, static_cast<const __nv_bfloat16*>(down), h->p.Dt, s)) !=
        cudaSuccess)
      break;
    if ((ce = mr::launch_dnorm(d, h->p.Dt, h->p.dnorm, s)) != cudaSuccess) break;
    st = mr::build_recovery_basis(d, h->p.Dt, h->p.U, h->p.eigvals, s, mr::take_prepare_stall());
    if (st != MOE_READER_OK) break;
    if ((ce = mr::launch_transpose_u(d, h->p.U, h->p.Ut, s)) != cudaSuccess) break;
    if ((ce = mr::launch_project_b(d, h->p.Dt, h->p.U, h->p.b, s)) != cudaSuccess) break;
    if ((ce = mr::launch_bnorm2(d, h->p.b, h->p.bnorm2, s)) != cudaSuccess) break;
    if ((ce = mr::configure_decode_kernels(d)) != cudaSuccess) break;
    h->grid = mr::decode_grid(d);
    if (h->grid <= 0) {
      ce = cudaErrorInvalidConfiguration;
      break;
    }
    ce = cudaStreamSynchronize(s);
  } while (0);
  if (ce != cudaSuccess || st != MOE_READER_OK) {
    cudaStreamSynchronize(s);
    cudaFree(pbase);
    cudaFree(wbase);
    free(h);
    return st != MOE_READER_OK ? st : cuda_status(ce);
  }
  *out = h;
  return MOE_READER_OK;
}

int moe_reader_decode(moe_reader_t* h, const float* x, int32_t B, const int32_t* expert_ids,
                      const float* expert_w, int32_t k, float* y, void* stream) {
  int st = check_decode_args(h, x, B, expert_ids, expert_w, k, y);
  if (st != MOE_READER_OK) return st;
  if (B == 0) return MOE_READER_OK;
  if (!aligned(x, 16) || !aligned(expert_ids, 16) || !aligned(expert_w, 16) || !aligned(y, 16))
    return MOE_READER_EINVAL;
  if ((const void*)x == (const void*)y) return MOE_READER_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t ce = launch_profiled(h, x, B, expert_ids, expert_w, k, y, s);
  h->inject = 0;
  if (ce != cudaSuccess) return cuda_status(ce);
  h->has_decode = 1;
  h->last_B = B;
  h->last_k = k;
  h->last_shared = 0;
  h->last_stream = s;
  return MOE_READER_OK;
}

int moe_reader_decode_shared(moe_reader_t* h, const float* x, int32_t B, const int32_t* expert_ids,
                             const float* expert_w, int32_t k, float* y, void* stream) {
  int st = check_decode_args(h, x, B, expert_ids, expert_w, k, y);
  if (st != MOE_READER_OK) return st;
  if (B == 0) return MOE_READER_OK;
  if (!aligned(x, 16) || !aligned(expert_ids, 16) || !aligned(expert_w, 16) || !aligned(y, 16))
    return MOE_READER_EINVAL;
  if ((const void*)x == (const void*)y) return MOE_READER_EINVAL;
  if (!mr::shared_supported(h->d, B)) return MOE_READER_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t ce = launch_profiled(h, x, B, expert_ids, expert_w, k, y, s, true);
  h->inject = 0;
  if (ce != cudaSuccess) return cuda_status(ce);
  h->has_decode = 1;
  h->last_B = B;
  h->last_k = k;
  h->last_shared = 1;
  h->last_stream = s;
  return MOE_READER_OK;
}

int moe_reader_get_kept_shared(moe_reader_t* h, int32_t* kept_host, int64_t capacity,
                               int32_t* count_out) {
  if (!h || (!kept_host && capacity > 0)) return MOE_READER_EINVAL;
  if (!h->has_decode || !h->last_shared) return MOE_READER_ESTATE;
  cudaStream_t s = h->last_stream;
  cudaError_t ce = cudaStreamSynchronize(s);
  if (ce != cudaSuccess) return cuda_status(ce);
  int32_t K = 0;
  if ((ce = cudaMemcpy(&K, h->ws.sK, 4, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_status(ce);
  if (count_out) *count_out = K;
  if (capacity < K) return MOE_READER_EINVAL;
  if (K > 0 && (ce = cudaMemcpy(kept_host, h->ws.skept, (size_t)K * 4, cudaMemcpyDeviceToHost)) !=
                   cudaSuccess)
    return cuda_status(ce);
  return MOE_READER_OK;
}

int moe_reader_decode_host(moe_reader_t* h, const float* x_host, int32_t B,
                           const int32_t* ids_host, const float* w_host, int32_t k,
                           float* y_host, void* stream) {
  int st = check_decode_args(h, x_host, B, ids_host, w_host, k, y_host);
  if (st != MOE_READER_OK) return st;
  if (B == 0) return MOE_READER_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Dims& d = h->d;
  cudaError_t ce;
  if ((ce = cudaMemcpyAsync(h->ws.x_stage, x_host, (size_t)B * d.H * 4, cudaMemcpyHostToDevice, s)) !=
      cudaSuccess)
    return cuda_status(ce);
  if ((ce = cudaMemcpyAsync(h->ws.ids_stage, ids_host, (size_t)B * d.topk * 4,
                            cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return cuda_status(ce);
  if ((ce = cudaMemcpyAsync(h->ws.w_stage, w_host, (size_t)B * d.topk * 4, cudaMemcpyHostToDevice,
                            s)) != cudaSuccess)
    return cuda_status(ce);
  ce = launch_profiled(h, h->ws.x_stage, B, h->ws.ids_stage, h->ws.w_stage, k, h->ws.y_stage, s);
  h->inject = 0;
  if (ce != cudaSuccess) return cuda_status(ce);
  h->has_decode = 1;
  h->last_B = B;
  h->last_k = k;
  h->last_shared = 0;
  h->last_stream = s;
  if ((ce = cudaMemcpyAsync(y_host, h->ws.y_stage, (size_t)B * d.H * 4, cudaMemcpyDeviceToHost, s)) !=
      cudaSuccess)
    return cuda_status(ce);
  uint32_t bits = 0;
  if ((ce = cudaMemcpyAsync(&bits, h->ws.err, 4, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_status(ce);
  if ((ce = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_status(ce);
  if (bits & mr::kErrTimeout) {
    cudaMemset(h->ws.sync, 0, mr::sync_words(d) * 4);
    cudaMemset(h->ws.err, 0, 4);
    return MOE_READER_ETIMEOUT;
  }
  if (bits) return MOE_READER_EDEVICE;
  return MOE_READER_OK;
}

int moe_reader_decode_stack(moe_reader_t* const* layers, int32_t L, const float* h_in, int32_t B,
                            const int32_t* expert_ids, const float* expert_w, int32_t k,
                            float* h_out, float* y_layers, void* stream) {
  if (!layers || L < 1) return MOE_READER_EINVAL;
  for (int l = 0; l < L; ++l) {
    const moe_reader* h = layers[l];
    if (!h) return MOE_READER_EINVAL;
    const mr::Dims& a = h->d;
    const mr::Dims& b = layers[0]->d;
    if (a.H != b.H || a.E != b.E || a.topk != b.topk || a.I != b.I || a.c != b.c || a.r != b.r ||
        h->device != layers[0]->device || h->grid != layers[0]->grid)
      return MOE_READER_EINVAL;
    if (B < 0 || B > a.Bmax) return MOE_READER_EINVAL;
    for (int m = 0; m < l; ++m)
      if (layers[m] == h) return MOE_READER_EINVAL;   // each layer needs its own counters
  }
  if (k < 0 || k > layers[0]->d.N) return MOE_READER_EINVAL;
  if (B == 0) return MOE_READER_OK;
  if (!h_in || !expert_ids || !expert_w || !h_out) return MOE_READER_EINVAL;
  if (!aligned(h_in, 16) || !aligned(expert_ids, 16) || !aligned(expert_w, 16) ||
      !aligned(h_out, 16) || !aligned(y_layers, 16))
    return MOE_READER_EINVAL;
  const size_t act = (size_t)B * layers[0]->d.H * 4;
  auto overlap = [](const void* p, size_t pn, const void* q, size_t qn) {
    const char* a = static_cast<const char*>(p);
    const char* b = static_cast<const char*>(q);
    return a < b + qn && b < a + pn;
  };
  if (overlap(h_in, act, h_out, act)) return MOE_READER_EINVAL;
  if (y_layers && (overlap(y_layers, act * L, h_in, act) || overlap(y_layers, act * L, h_out, act)))
    return MOE_READER_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t ce =
      mr::launch_decode_stack(layers, L, h_in, B, expert_ids, expert_w, k, h_out, y_layers, s);
  for (int l = 0; l < L; ++l) layers[l]->inject = 0;
  if (ce != cudaSuccess) return cuda_status(ce);
  for (int l = 0; l < L; ++l) {
    layers[l]->has_decode = 1;
    layers[l]->last_B = B;
    layers[l]->last_k = k;
    layers[l]->last_shared = 0;
    layers[l]->last_stream = s;
  }
  return MOE_READER_OK;
}

int moe_reader_set_wait_limit(moe_reader_t* h, uint64_t ns) {
  if (!h) return MOE_READER_EINVAL;
  h->wait_ns = ns;
  return MOE_READER_OK;
}

int moe_reader_inject_fault(moe_reader_t* h, uint32_t what) {
  const uint32_t handle_bits = MOE_READER_INJECT_DECODE_STALL;
  const uint32_t global_bits = MOE_READER_INJECT_PREPARE_STALL | MOE_READER_INJECT_ALLOC_FAIL;
  if (what == 0 || (what & ~(handle_bits | global_bits))) return MOE_READER_EINVAL;
  if (h ? (what & global_bits) != 0 : (what & handle_bits) != 0) return MOE_READER_EINVAL;
  if (h) {
    h->inject |= what;
    return MOE_READER_OK;
  }
  if (what & MOE_READER_INJECT_PREPARE_STALL) g_stall_next_prepare.store(1);
  if (what & MOE_READER_INJECT_ALLOC_FAIL) g_fail_next_alloc.store(1);
  return MOE_READER_OK;
}

int moe_reader_status(moe_reader_t* h, uint32_t* bits_out) {
  if (!h) return MOE_READER_EINVAL;
  cudaError_t ce = h->has_decode ? cudaStreamSynchronize(h->last_stream) : cudaDeviceSynchronize();
  if (ce != cudaSuccess) return cuda_status(ce);
  uint32_t bits = 0;
  if ((ce = cudaMemcpy(&bits, h->ws.err, 4, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_status(ce);
  if ((ce = cudaMemset(h->ws.err, 0, 4)) != cudaSuccess) return cuda_status(ce);
  if (bits & mr::kErrTimeout) {
    // a timed-out decode leaves its counters behind: clear them for the next call
    if ((ce = cudaMemset(h->ws.sync, 0, mr::sync_words(h->d) * 4)) != cudaSuccess)
      return cuda_status(ce);
  }
  if (bits_out) *bits_out = bits;
  if (bits & mr::kErrTimeout) return MOE_READER_ETIMEOUT;
  if (bits) return MOE_READER_EDEVICE;
  return MOE_READER_OK;
}

int moe_reader_get_stats(moe_reader_t* h, moe_reader_stats* out) {
  if (!h || !out) return MOE_READER_EINVAL;
  if (!h->has_decode) return MOE_READER_ESTATE;
  const Dims& d = h->d;
  cudaStream_t s = h->last_stream;
  cudaError_t ce = mr::launch_stats(*h, h->last_B, h->last_k, s);
  if (ce != cudaSuccess) return cuda_status(ce);
  unsigned long long c[16];
  if ((ce = cudaMemcpyAsync(c, h->ws.counters, sizeof(c), cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_status(ce);
  if ((ce = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_status(ce);
  memset(out, 0, sizeof(*out));
  auto up = [](unsigned long long bytes) { return (bytes + 31) / 32; };
  const unsigned long long runs = c[0], kept = c[1], skipped = c[2], experts = c[3], bsec = c[4];
  const int B = h->last_B;
  out->sectors[MOE_READER_ARR_CODES] =
      runs * 2 * up((unsigned long long)(d.trit5 ? (d.I + 4) / 5 : (d.I + 3) / 4));
  out->sectors[MOE_READER_ARR_SCALES] = experts * d.nb * up(2ULL * d.I * 2);
  out->sectors[MOE_READER_ARR_DNORM] = experts * up(4ULL * d.I);
  out->sectors[MOE_READER_ARR_G] = kept * up(2ULL * d.H);
  out->sectors[MOE_READER_ARR_V] = kept * up(2ULL * d.H);
  out->sectors[MOE_READER_ARR_DT] = kept * up(2ULL * d.H);
  out->sectors[MOE_READER_ARR_B] = bsec;
  out->sectors[MOE_READER_ARR_U] = skipped ? up(2ULL * d.H * d.r) : 0;
  out->dense_sectors = experts * 3 * up(2ULL * d.I * d.H);
  out->activation_bytes = (unsigned long long)B * d.H * 4 * 2 + (unsigned long long)B * d.topk * 8;
  out->batch = B;
  out->k = h->last_k;
  return MOE_READER_OK;
}

int moe_reader_get_kept(moe_reader_t* h, int32_t* kept_host, int64_t capacity) {
  if (!h || (!kept_host && capacity > 0)) return MOE_READER_EINVAL;
  if (!h->has_decode || h->last_shared) return MOE_READER_ESTATE;
  const int B = h->last_B, k = h->last_k;
  const int64_t n = (int64_t)B * k;
  if (capacity < n) return MOE_READER_EINVAL;
  if (n == 0) return MOE_READER_OK;
  cudaStream_t s = h->last_stream;
  int32_t* dev = nullptr;
  cudaError_t ce = mr::device_alloc(reinterpret_cast<void**>(&dev), (size_t)n * 4);
  if (ce != cudaSuccess) return cuda_status(ce);
  do {
    if ((ce = mr::launch_gather_kept(*h, B, k, dev, s)) != cudaSuccess) break;
    if ((ce = cudaMemcpyAsync(kept_host, dev, (size_t)n * 4, cudaMemcpyDeviceToHost, s)) !=
        cudaSuccess)
      break;
    ce = cudaStreamSynchronize(s);
  } while (0);
  cudaFree(dev);
  if (ce != cudaSuccess) return cuda_status(ce);
  for (int t = 0; t < B; ++t) std::sort(kept_host + (int64_t)t * k, kept_host + (int64_t)(t + 1) * k);
  return MOE_READER_OK;
}

int64_t moe_reader_export_size(moe_reader_t* h, int32_t which) {
  if (!h) return MOE_READER_EINVAL;
  return export_size(h, which);
}

int moe_reader_export(moe_reader_t* h, int32_t which, void* dst, int64_t bytes) {
  if (!h || !dst) return MOE_READER_EINVAL;
  const int64_t need = export_size(h, which);
  if (need < 0) return (int)need;
  if (bytes != need) return MOE_READER_EINVAL;
  cudaError_t ce = cudaDeviceSynchronize();
  if (ce != cudaSuccess) return cuda_status(ce);
  ce = cudaMemcpy(dst, export_ptr(h, which), (size_t)need, cudaMemcpyDeviceToHost);
  return cuda_status(ce);
}

int moe_reader_get_info(moe_reader_t* h, moe_reader_info* out) {
  if (!h || !out) return MOE_READER_EINVAL;
  memset(out, 0, sizeof(*out));
  out->hidden_padded = h->d.Hp;
  out->num_blocks = h->d.nb;
  out->routed_channels = h->d.N;
  out->run_stride = h->d.S;
  for (int i = 0; i < 9; ++i) out->resident_bytes[i] = h->resident[i];
  return MOE_READER_OK;
}

int moe_reader_set_profiling(moe_reader_t* h, int32_t enable) {
  if (!h) return MOE_READER_EINVAL;
  if (enable && !h->prof_created) {
    for (int i = 0; i < mr::kProfSlots; ++i)
      for (int j = 0; j < 2; ++j) {
        const cudaError_t ce = cudaEventCreate(&h->prof_ev[i][j]);
        if (ce != cudaSuccess) return cuda_status(ce);
      }
    const cudaError_t ce = mr::device_alloc(
        reinterpret_cast<void**>(&h->prof_stamps),
        (size_t)mr::kProfSlots * h->grid * 5 * sizeof(unsigned long long));
    if (ce != cudaSuccess) return cuda_status(ce);
    h->prof_created = 1;
  }
  h->prof_on = enable ? 1 : 0;
  h->prof_used = 0;
  return MOE_READER_OK;
}

int moe_reader_read_profile(moe_reader_t* h, double* ms_out, int64_t capacity,
                            int64_t* calls_out) {
  if (!h || (!ms_out && capacity > 0)) return MOE_READER_EINVAL;
  const int used = h->prof_used < mr::kProfSlots ? h->prof_used : mr::kProfSlots;
  if (calls_out) *calls_out = used;
  if (capacity < used) return MOE_READER_EINVAL;
  if (used == 0) return MOE_READER_OK;
  std::vector<unsigned long long> st((size_t)used * h->grid * 5);
  for (int i = 0; i < used; ++i) {
    const cudaError_t ce = cudaEventSynchronize(h->prof_ev[i][1]);
    if (ce != cudaSuccess) return cuda_status(ce);
  }
  cudaError_t ce = cudaMemcpy(st.data(), h->prof_stamps, st.size() * sizeof(unsigned long long),
                              cudaMemcpyDeviceToHost);
  if (ce != cudaSuccess) return cuda_status(ce);
  for (int i = 0; i < used; ++i) {
    float ms = 0.f;
    ce = cudaEventElapsedTime(&ms, h->prof_ev[i][0], h->prof_ev[i][1]);
    if (ce != cudaSuccess) return cuda_status(ce);
    double* row = ms_out + (size_t)i * mr::kPhases;
    row[0] = ms;
    // phase boundaries: the earliest start, then the latest end of each phase
    unsigned long long t0 = ~0ull, e[4] = {0, 0, 0, 0};
    for (int c = 0; c < h->grid; ++c) {
      const unsigned long long* r = &st[((size_t)i * h->grid + c) * 5];
      t0 = std::min(t0, r[0]);
      for (int q = 0; q < 4; ++q) e[q] = std::max(e[q], r[q + 1]);
    }
    unsigned long long prev = t0;
    for (int q = 0; q < 4; ++q) {
      row[q + 1] = e[q] > prev ? (double)(e[q] - prev) * 1e-6 : 0.0;
      prev = std::max(prev, e[q]);
    }
  }
  return MOE_READER_OK;
}

void moe_reader_destroy(moe_reader_t* h) {
  if (!h) return;
  cudaDeviceSynchronize();
  if (h->prof_created) {
    for (int i = 0; i < mr::kProfSlots; ++i)
      for (int j = 0; j < 2; ++j) cudaEventDestroy(h->prof_ev[i][j]);
    cudaFree(h->prof_stamps);
  }
  free_handle_memory(h);
  free(h);
}

}  // extern "C"
