// C ABI of libsdpa.so: argument validation, kernel-family choice and launches.
// The operation and every convention are documented in include/sdpa.h.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include "launch.h"
#include "../../include/sdpa.h"

namespace sdpa {
namespace {

__device__ unsigned g_device_error = 0;

std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_path{SDPA_PATH_AUTO};
std::atomic<int> g_inject{0};
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};

constexpr int kMaxDevices = 64;
std::atomic<unsigned*> g_err_ptr[kMaxDevices];
std::mutex g_err_mu;

// Device address of the error word on the current device, looked up once per device (the
// library assumes each device's primary context and no device reset while it is loaded).
// Several host threads may call this at once.
int error_word(unsigned** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SDPA_ERR_CUDA;
  unsigned* ptr = g_err_ptr[dev].load();
  if (!ptr) {
    std::lock_guard<std::mutex> lock(g_err_mu);
    ptr = g_err_ptr[dev].load();
    if (!ptr) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_device_error) != cudaSuccess || !addr) return SDPA_ERR_CUDA;
      ptr = static_cast<unsigned*>(addr);
      g_err_ptr[dev].store(ptr);
    }
  }
  *out = ptr;
  return SDPA_OK;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }
bool aligned4(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

size_t elem_size(int dtype) { return dtype == SDPA_F32 ? 4 : 2; }

sdpa_layout_t contiguous(int H, int L, int D) {
  return sdpa_layout_t{(int64_t)H * L * D, (int64_t)L * D, (int64_t)D};
}

sdpa_strides_t contiguous_strides(int Hq, int Hkv, int Lq, int Lkv, int D) {
  const sdpa_layout_t lq = contiguous(Hq, Lq, D), lk = contiguous(Hkv, Lkv, D);
  return sdpa_strides_t{lq, lk, lk, lq, lq, lq, lk, lk};
}

// Validates the layout of one [B, H, L, D] tensor (strides positive, multiples of 16
// bytes, no two elements at one address: sorted by stride, each stride covers the extent
// of the smaller dimensions) and returns its byte extent in *bytes.
bool check_layout(const sdpa_layout_t& l, int B, int H, int L, int D, size_t es, Layout* out, size_t* bytes) {
  const int64_t st[3] = {l.batch, l.head, l.row};
  const int64_t n[3] = {B, H, L};
  for (int a = 0; a < 3; ++a)
    if (st[a] < 1 || (st[a] * (int64_t)es) % 16 != 0 || st[a] > ((int64_t)1 << 40)) return false;
  int order[3] = {0, 1, 2};
  for (int a = 0; a < 3; ++a)
    for (int c = a + 1; c < 3; ++c)
      if (st[order[c]] < st[order[a]]) std::swap(order[a], order[c]);
  int64_t covered = D;  // extent of the dimensions below, in elements
  for (int a = 0; a < 3; ++a) {
    const int dim = order[a];
    if (n[dim] == 1) continue;
    if (st[dim] < covered) return false;
    covered = st[dim] * (n[dim] - 1) + covered;
  }
  *bytes = (size_t)(((int64_t)(B - 1) * l.batch + (int64_t)(H - 1) * l.head + (int64_t)(L - 1) * l.row + D) *
                    (int64_t)es);
  *out = Layout{l.batch, l.head, l.row};
  return true;
}

// Validates an attention mask (kind, alignment, strides) and fills p->mask, mask_kind and
// lm; *bytes is the byte extent the kernels may read (each row up to the next multiple of
// 16 bytes past Lkv), 0 without a mask.
bool check_mask(const sdpa_mask_t* m, int dtype, Problem* p, size_t* bytes) {
  *bytes = 0;
  if (!m || m->kind == SDPA_MASK_NONE) return true;
  if (m->kind != SDPA_MASK_BOOL && m->kind != SDPA_MASK_ADDITIVE) return false;
  if (!m->ptr || !aligned16(m->ptr)) return false;
  const int64_t es = m->kind == SDPA_MASK_BOOL ? 1 : (int64_t)elem_size(dtype);
  const int64_t st[3] = {m->batch, m->head, m->row};
  for (int a = 0; a < 3; ++a)
    if (st[a] < 0 || (st[a] * es) % 16 != 0 || st[a] > ((int64_t)1 << 40)) return false;
  const int64_t row_bytes = ((int64_t)p->Lkv * es + 15) / 16 * 16;
  *bytes = (size_t)(((int64_t)(p->B - 1) * m->batch + (int64_t)(p->Hq - 1) * m->head + (int64_t)(p->Lq - 1) * m->row) * es +
                    row_bytes);
  p->mask = m->ptr;
  p->mask_kind = m->kind;
  p->lm = Layout{m->batch, m->head, m->row};
  return true;
}

// Checks sizes, dtype and scale; fills the size fields of *p.
int check_sizes(int B, int Hq, int Hkv, int Lq, int Lkv, int D, float scale, int dtype,
                Problem* p) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Lq < 1 || Lkv < 1 || D < 1) return SDPA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return SDPA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return SDPA_ERR_INVALID_ARG;
  if (dtype != SDPA_F32 && dtype != SDPA_F16 && dtype != SDPA_BF16) return SDPA_ERR_UNSUPPORTED;
  if (D != 32 && D != 64 && D != 96 && D != 128 && D != 256) return SDPA_ERR_UNSUPPORTED;
  if (B > 65535 || Hq > 65535) return SDPA_ERR_UNSUPPORTED;
  // Keep every element index comfortably inside int64 (and far above any real HBM size).
  const double qe = (double)B * Hq * Lq * D, ke = (double)B * Hkv * Lkv * D;
  if (qe > 4.0e12 || ke > 4.0e12) return SDPA_ERR_UNSUPPORTED;
  std::memset(p, 0, sizeof(*p));
  p->B = B;
  p->Hq = Hq;
  p->Hkv = Hkv;
  p->Lq = Lq;
  p->Lkv = Lkv;
  p->D = D;
  p->G = Hq / Hkv;
  p->scale = scale;
  p->scale_log2 = scale * kLog2e;
  p->wait_limit_ns = g_wait_limit_ns.load();
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    p->num_sms = 0;  // no prefetch hints
  return SDPA_OK;
}

// Causal mode: none, top-left (key j hidden from query i when j > i) or bottom-right
// (hidden when j > i + Lkv - Lq; needs Lq <= Lkv so that every query sees key 0).
int set_causal(Problem* p, int is_causal) {
  if (is_causal < SDPA_CAUSAL_NONE || is_causal > SDPA_CAUSAL_BOTTOM_RIGHT) return SDPA_ERR_INVALID_ARG;
  p->causal = is_causal != SDPA_CAUSAL_NONE ? 1 : 0;
  p->coff = 0;
  if (is_causal == SDPA_CAUSAL_BOTTOM_RIGHT) {
    if (p->Lq > p->Lkv) return SDPA_ERR_UNSUPPORTED;
    p->coff = p->Lkv - p->Lq;
  }
  return SDPA_OK;
}

enum class Family { kTensor, kSimt, kVector };

int choose(const Problem& p, int dtype, Family* f) {
  const int forced = g_path.load();
  switch (forced) {
    case SDPA_PATH_TENSOR:
      if (!tensor_supported(p, dtype)) return SDPA_ERR_UNSUPPORTED;
      *f = Family::kTensor;
      return SDPA_OK;
    case SDPA_PATH_SIMT:
      *f = Family::kSimt;
      return SDPA_OK;
    case SDPA_PATH_VECTOR:
      if (!vector_supported(p, dtype)) return SDPA_ERR_UNSUPPORTED;
      *f = Family::kVector;
      return SDPA_OK;
    default:
      break;
  }
  if (vector_supported(p, dtype)) *f = Family::kVector;
  else if (tensor_supported(p, dtype)) *f = Family::kTensor;
  else *f = Family::kSimt;
  return SDPA_OK;
}

// ---- optional per-kernel device timing (CUDA events bracketing each launch) ----
struct EventPair {
  cudaEvent_t start = nullptr, stop = nullptr;
};
struct PendingTiming {
  int kernel;
  EventPair ev;
};
std::mutex g_timing_mu;
std::atomic<bool> g_timing_on{false};
std::vector<EventPair> g_event_pool;
std::vector<PendingTiming> g_pending;
double g_total_ms[SDPA_KERNEL_COUNT] = {};
uint64_t g_timed_launches[SDPA_KERNEL_COUNT] = {};

bool take_pair(EventPair* ev) {
  std::lock_guard<std::mutex> lock(g_timing_mu);
  if (!g_event_pool.empty()) {
    *ev = g_event_pool.back();
    g_event_pool.pop_back();
    return true;
  }
  if (cudaEventCreate(&ev->start) != cudaSuccess) return false;
  if (cudaEventCreate(&ev->stop) != cudaSuccess) {
    cudaEventDestroy(ev->start);
    return false;
  }
  return true;
}

// Launches one kernel through `fn`, counting it and, when timing is on, bracketing it with
// events on its stream.
template <typename Fn>
cudaError_t launch_one(int kernel, cudaStream_t s, Fn fn) {
  EventPair ev;
  const bool timed = g_timing_on.load() && take_pair(&ev);
  if (timed) cudaEventRecord(ev.start, s);
  cudaError_t e = fn();
  if (e == cudaSuccess) g_launches.fetch_add(1);
  if (timed) {
    cudaEventRecord(ev.stop, s);
    std::lock_guard<std::mutex> lock(g_timing_mu);
    if (e == cudaSuccess) g_pending.push_back({kernel, ev});
    else g_event_pool.push_back(ev);
  }
  return e;
}

int status_of(cudaError_t e) { return e == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA; }

// ---- fork / join of the two tiled backward kernels ----
// The dK/dV and dQ kernels both need only δ, so they run concurrently: the dK/dV kernel on
// a library-owned stream of the highest priority (its pending blocks are scheduled first),
// the dQ kernel on the caller's stream, whose blocks fill the SMs that the tail of the
// dK/dV grid leaves idle.  Events order the side stream after the caller's earlier work
// and the caller's stream after the dK/dV kernel, so the call stays ordered on the
// caller's stream like any single-stream launch sequence (graph capture follows the fork
// into the side stream and back).  One side stream and one event pair per device; the
// record / wait / launch sequence holds a mutex so that concurrent host threads cannot
// interleave their events.
struct Fork {
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
Fork g_fork[kMaxDevices];
std::mutex g_fork_mu;

// Side stream and events of the current device, created on first use (caller holds
// g_fork_mu).
cudaError_t fork_of_device(Fork** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  Fork& f = g_fork[dev];
  if (!f.side) {
    int least = 0, greatest = 0;
    if ((e = cudaDeviceGetStreamPriorityRange(&least, &greatest)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&f.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&f.join, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithPriority(&f.side, cudaStreamNonBlocking, greatest)) != cudaSuccess) {
      f.side = nullptr;
      return e;
    }
  }
  *out = &f;
  return cudaSuccess;
}

}  // namespace
}  // namespace sdpa

using namespace sdpa;

extern "C" int sdpa_fwd_masked(const void* q, const void* k, const void* v, void* out, float* lse,
                               const float* sinks, const sdpa_mask_t* mask, int B, int Hq, int Hkv,
                               int Lq, int Lkv, int D, float scale, int is_causal, int dtype,
                               const sdpa_strides_t* strides, void* stream) {
  Problem p;
  int st = check_sizes(B, Hq, Hkv, Lq, Lkv, D, scale, dtype, &p);
  if (st != SDPA_OK) return st;
  if (!q || !k || !v || !out || !strides) return SDPA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse) ||
      !aligned4(sinks))
    return SDPA_ERR_INVALID_ARG;
  const size_t es = elem_size(dtype);
  size_t qb, kb, vb, ob;
  if (!check_layout(strides->q, B, Hq, Lq, D, es, &p.lq, &qb) || !check_layout(strides->k, B, Hkv, Lkv, D, es, &p.lk, &kb) ||
      !check_layout(strides->v, B, Hkv, Lkv, D, es, &p.lv, &vb) || !check_layout(strides->o, B, Hq, Lq, D, es, &p.lo, &ob))
    return SDPA_ERR_INVALID_ARG;
  const size_t lb = lse ? (size_t)B * Hq * Lq * sizeof(float) : 0;
  if (overlaps(out, ob, q, qb) || overlaps(out, ob, k, kb) || overlaps(out, ob, v, vb) ||
      overlaps(lse, lb, q, qb) || overlaps(lse, lb, k, kb) || overlaps(lse, lb, v, vb) ||
      overlaps(lse, lb, out, ob))
    return SDPA_ERR_INVALID_ARG;
  const size_t sb = (size_t)Hq * sizeof(float);
  if (overlaps(out, ob, sinks, sb) || overlaps(lse, lb, sinks, sb)) return SDPA_ERR_INVALID_ARG;
  size_t mb;
  if (!check_mask(mask, dtype, &p, &mb)) return SDPA_ERR_INVALID_ARG;
  if (overlaps(out, ob, p.mask, mb) || overlaps(lse, lb, p.mask, mb)) return SDPA_ERR_INVALID_ARG;
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.lse = lse;
  p.sinks = sinks;
  if ((st = set_causal(&p, is_causal)) != SDPA_OK) return st;
  Family f;
  if ((st = choose(p, dtype, &f)) != SDPA_OK) return st;
  if ((st = error_word(&p.err)) != SDPA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (f) {
    case Family::kVector:
      e = launch_one(SDPA_KERNEL_VEC_FWD, s, [&] {
        return vector_mma_supported(p, dtype) ? launch_vector_mma_fwd(p, dtype, s) : launch_vector_fwd(p, dtype, s);
      });
      break;
    case Family::kTensor:
      p.inject = g_inject.exchange(0);
      e = launch_one(SDPA_KERNEL_FWD, s, [&] { return launch_tc_fwd(p, dtype, s); });
      break;
    default:
      e = launch_one(SDPA_KERNEL_FWD, s, [&] { return launch_simt_fwd(p, dtype, s); });
      break;
  }
  return status_of(e);
}

extern "C" int sdpa_fwd_sinks(const void* q, const void* k, const void* v, void* out, float* lse,
                              const float* sinks, int B, int Hq, int Hkv, int Lq, int Lkv, int D,
                              float scale, int is_causal, int dtype, const sdpa_strides_t* strides,
                              void* stream) {
  return sdpa_fwd_masked(q, k, v, out, lse, sinks, nullptr, B, Hq, Hkv, Lq, Lkv, D, scale, is_causal,
                         dtype, strides, stream);
}

extern "C" int sdpa_fwd_strided(const void* q, const void* k, const void* v, void* out, float* lse,
                                int B, int Hq, int Hkv, int Lq, int Lkv, int D, float scale,
                                int is_causal, int dtype, const sdpa_strides_t* strides, void* stream) {
  return sdpa_fwd_sinks(q, k, v, out, lse, nullptr, B, Hq, Hkv, Lq, Lkv, D, scale, is_causal, dtype,
                        strides, stream);
}

extern "C" int sdpa_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                        int B, int Hq, int Hkv, int Lq, int Lkv, int D, float scale,
                        int is_causal, int dtype, void* stream) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Lq < 1 || Lkv < 1 || D < 1) return SDPA_ERR_INVALID_ARG;
  const sdpa_strides_t st = contiguous_strides(Hq, Hkv, Lq, Lkv, D);
  return sdpa_fwd_strided(q, k, v, out, lse, B, Hq, Hkv, Lq, Lkv, D, scale, is_causal, dtype, &st, stream);
}

extern "C" size_t sdpa_bwd_workspace_size(int B, int Hq, int Hkv, int Lq, int Lkv, int D,
                                          int dtype) {
  Problem p;
  if (check_sizes(B, Hq, Hkv, Lq, Lkv, D, 1.0f, dtype, &p) != SDPA_OK) return 0;
  const size_t bytes = (size_t)B * Hq * Lq * sizeof(float);
  return (bytes + 255) / 256 * 256;
}

extern "C" int sdpa_bwd_masked(const void* q, const void* k, const void* v, const void* out,
                               const void* dout, const float* lse, const float* sinks,
                               const sdpa_mask_t* mask, void* dq, void* dk, void* dv, float* dsinks,
                               int B, int Hq, int Hkv, int Lq, int Lkv, int D, float scale,
                               int is_causal, int dtype, const sdpa_strides_t* strides,
                               void* workspace, size_t workspace_bytes, void* stream) {
  Problem p;
  int st = check_sizes(B, Hq, Hkv, Lq, Lkv, D, scale, dtype, &p);
  if (st != SDPA_OK) return st;
  if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv || !strides) return SDPA_ERR_INVALID_ARG;
  if (dsinks && !sinks) return SDPA_ERR_INVALID_ARG;
  const void* all[] = {q, k, v, out, dout, lse, dq, dk, dv};
  for (const void* ptr : all)
    if (!aligned16(ptr)) return SDPA_ERR_INVALID_ARG;
  if (!aligned4(sinks) || !aligned4(dsinks)) return SDPA_ERR_INVALID_ARG;
  const size_t need = sdpa_bwd_workspace_size(B, Hq, Hkv, Lq, Lkv, D, dtype);
  if (!workspace || workspace_bytes < need) return SDPA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return SDPA_ERR_INVALID_ARG;
  const size_t es = elem_size(dtype);
  size_t qb, kb, vb, ob, dob, dqb, dkb, dvb;
  if (!check_layout(strides->q, B, Hq, Lq, D, es, &p.lq, &qb) || !check_layout(strides->k, B, Hkv, Lkv, D, es, &p.lk, &kb) ||
      !check_layout(strides->v, B, Hkv, Lkv, D, es, &p.lv, &vb) || !check_layout(strides->o, B, Hq, Lq, D, es, &p.lo, &ob) ||
      !check_layout(strides->dout, B, Hq, Lq, D, es, &p.ldo, &dob) ||
      !check_layout(strides->dq, B, Hq, Lq, D, es, &p.ldq, &dqb) ||
      !check_layout(strides->dk, B, Hkv, Lkv, D, es, &p.ldk, &dkb) ||
      !check_layout(strides->dv, B, Hkv, Lkv, D, es, &p.ldv, &dvb))
    return SDPA_ERR_INVALID_ARG;
  const size_t lb = (size_t)B * Hq * Lq * sizeof(float), sb = (size_t)Hq * sizeof(float);
  size_t mb;
  if (!check_mask(mask, dtype, &p, &mb)) return SDPA_ERR_INVALID_ARG;
  const void* ins[] = {q, k, v, out, dout, lse, sinks, p.mask};
  const size_t in_bytes[] = {qb, kb, vb, ob, dob, lb, sb, mb};
  void* outs[] = {dq, dk, dv, workspace, dsinks};
  const size_t out_bytes[] = {dqb, dkb, dvb, need, sb};
  for (int a = 0; a < 5; ++a) {
    for (int c = 0; c < 8; ++c)
      if (overlaps(outs[a], out_bytes[a], ins[c], in_bytes[c])) return SDPA_ERR_INVALID_ARG;
    for (int c = a + 1; c < 5; ++c)
      if (overlaps(outs[a], out_bytes[a], outs[c], out_bytes[c])) return SDPA_ERR_INVALID_ARG;
  }
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = out;
  p.dout = dout;
  p.lse = const_cast<float*>(lse);
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.delta = static_cast<float*>(workspace);
  p.sinks = sinks;
  p.dsinks = dsinks;
  if ((st = set_causal(&p, is_causal)) != SDPA_OK) return st;
  Family f;
  if ((st = choose(p, dtype, &f)) != SDPA_OK) return st;
  if ((st = error_word(&p.err)) != SDPA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  // The short-query backward computes δ inside its own kernel; the sink gradients need it
  // in the workspace, so then the δ pre-pass runs for them.
  if (f != Family::kVector || dsinks) {
    e = launch_one(SDPA_KERNEL_DELTA, s, [&] { return launch_delta(p, dtype, s); });
    if (e != cudaSuccess) return status_of(e);
  }
  if (dsinks) {
    e = launch_one(SDPA_KERNEL_SINK_GRAD, s, [&] { return launch_sink_grad(p, s); });
    if (e != cudaSuccess) return status_of(e);
  }
  if (f == Family::kVector)
    return status_of(launch_one(SDPA_KERNEL_VEC_BWD, s, [&] {
      return vector_mma_supported(p, dtype) ? launch_vector_mma_bwd(p, dtype, s) : launch_vector_bwd(p, dtype, s);
    }));
  const bool tc256 = f == Family::kTensor && tensor_bwd256_supported(p, dtype);
  const bool tc = tc256 || (f == Family::kTensor && tensor_bwd_supported(p, dtype));
  if (f == Family::kTensor && !tc && g_path.load() == SDPA_PATH_TENSOR) return SDPA_ERR_UNSUPPORTED;
  auto launch_dkdv = [&](cudaStream_t st) {
    return launch_one(SDPA_KERNEL_DKDV, st, [&] {
      if (!tc) return launch_simt_dkdv(p, dtype, st);
      return tc256 ? launch_tc_dkdv256(p, dtype, st) : launch_tc_dkdv(p, dtype, st);
    });
  };
  auto launch_dq = [&](cudaStream_t st) {
    return launch_one(SDPA_KERNEL_DQ, st, [&] {
      if (!tc) return launch_simt_dq(p, dtype, st);
      return tc256 ? launch_tc_dq256(p, dtype, st) : launch_tc_dq(p, dtype, st);
    });
  };
  // While per-kernel timing is on, each kernel runs alone so that its events bracket only
  // its own work.
  if (!tc || g_timing_on.load()) {
    if ((e = launch_dkdv(s)) != cudaSuccess) return status_of(e);
    return status_of(launch_dq(s));
  }
  std::lock_guard<std::mutex> lock(g_fork_mu);
  Fork* fk = nullptr;
  if ((e = fork_of_device(&fk)) != cudaSuccess) return status_of(e);
  if ((e = cudaEventRecord(fk->fork, s)) != cudaSuccess) return status_of(e);
  if ((e = cudaStreamWaitEvent(fk->side, fk->fork, 0)) != cudaSuccess) return status_of(e);
  const cudaError_t e_kv = launch_dkdv(fk->side);
  const cudaError_t e_q = launch_dq(s);
  // The join is recorded and waited for even if a launch failed, so that the side stream
  // is always joined back (and released from any capture).
  e = cudaEventRecord(fk->join, fk->side);
  const cudaError_t e_join = e == cudaSuccess ? cudaStreamWaitEvent(s, fk->join, 0) : e;
  if (e_kv != cudaSuccess) return status_of(e_kv);
  if (e_q != cudaSuccess) return status_of(e_q);
  return status_of(e_join);
}

extern "C" int sdpa_bwd_sinks(const void* q, const void* k, const void* v, const void* out,
                              const void* dout, const float* lse, const float* sinks, void* dq,
                              void* dk, void* dv, float* dsinks, int B, int Hq, int Hkv, int Lq,
                              int Lkv, int D, float scale, int is_causal, int dtype,
                              const sdpa_strides_t* strides, void* workspace, size_t workspace_bytes,
                              void* stream) {
  return sdpa_bwd_masked(q, k, v, out, dout, lse, sinks, nullptr, dq, dk, dv, dsinks, B, Hq, Hkv, Lq, Lkv,
                         D, scale, is_causal, dtype, strides, workspace, workspace_bytes, stream);
}

extern "C" int sdpa_bwd_strided(const void* q, const void* k, const void* v, const void* out,
                                const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                int B, int Hq, int Hkv, int Lq, int Lkv, int D, float scale,
                                int is_causal, int dtype, const sdpa_strides_t* strides,
                                void* workspace, size_t workspace_bytes, void* stream) {
  return sdpa_bwd_sinks(q, k, v, out, dout, lse, nullptr, dq, dk, dv, nullptr, B, Hq, Hkv, Lq, Lkv, D,
                        scale, is_causal, dtype, strides, workspace, workspace_bytes, stream);
}

extern "C" int sdpa_bwd(const void* q, const void* k, const void* v, const void* out,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv,
                        int B, int Hq, int Hkv, int Lq, int Lkv, int D, float scale,
                        int is_causal, int dtype, void* workspace, size_t workspace_bytes,
                        void* stream) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Lq < 1 || Lkv < 1 || D < 1) return SDPA_ERR_INVALID_ARG;
  const sdpa_strides_t st = contiguous_strides(Hq, Hkv, Lq, Lkv, D);
  return sdpa_bwd_strided(q, k, v, out, dout, lse, dq, dk, dv, B, Hq, Hkv, Lq, Lkv, D, scale, is_causal,
                          dtype, &st, workspace, workspace_bytes, stream);
}

extern "C" int sdpa_poll_status(void* stream) {
  unsigned* err = nullptr;
  int st = error_word(&err);
  if (st != SDPA_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SDPA_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return SDPA_ERR_CUDA;
  if (word == 0) return SDPA_OK;
  const unsigned zero = 0;
  if (cudaMemcpy(err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return SDPA_ERR_CUDA;
  return SDPA_ERR_DEVICE_TIMEOUT;
}

extern "C" const char* sdpa_status_string(int status) {
  switch (status) {
    case SDPA_OK: return "ok";
    case SDPA_ERR_INVALID_ARG: return "invalid argument";
    case SDPA_ERR_UNSUPPORTED: return "unsupported dtype, head dim or shape";
    case SDPA_ERR_CUDA: return "CUDA error";
    case SDPA_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait timed out";
    case SDPA_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

extern "C" int sdpa_set_path(int path) {
  if (path < SDPA_PATH_AUTO || path > SDPA_PATH_VECTOR) return SDPA_ERR_INVALID_ARG;
  g_path.store(path);
  return SDPA_OK;
}

extern "C" uint64_t sdpa_launch_count(void) { return g_launches.load(); }

extern "C" int sdpa_timing_enable(int on) {
  g_timing_on.store(on != 0);
  return SDPA_OK;
}

extern "C" int sdpa_timing_read(int kernel, double* total_ms, uint64_t* launches) {
  if (kernel < 0 || kernel >= SDPA_KERNEL_COUNT || !total_ms || !launches) return SDPA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_timing_mu);
  int st = SDPA_OK;
  for (PendingTiming& pt : g_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(pt.ev.stop) != cudaSuccess ||
        cudaEventElapsedTime(&ms, pt.ev.start, pt.ev.stop) != cudaSuccess) {
      st = SDPA_ERR_CUDA;
    } else {
      g_total_ms[pt.kernel] += ms;
      g_timed_launches[pt.kernel] += 1;
    }
    g_event_pool.push_back(pt.ev);
  }
  g_pending.clear();
  *total_ms = g_total_ms[kernel];
  *launches = g_timed_launches[kernel];
  return st;
}

extern "C" void sdpa_timing_reset(void) {
  std::lock_guard<std::mutex> lock(g_timing_mu);
  for (PendingTiming& pt : g_pending) {
    cudaEventSynchronize(pt.ev.stop);
    g_event_pool.push_back(pt.ev);
  }
  g_pending.clear();
  for (int k = 0; k < SDPA_KERNEL_COUNT; ++k) {
    g_total_ms[k] = 0.0;
    g_timed_launches[k] = 0;
  }
}

extern "C" int sdpa_debug_inject_timeout(int on, uint64_t wait_limit_ns) {
  if (wait_limit_ns == 0) return SDPA_ERR_INVALID_ARG;
  g_inject.store(on ? 1 : 0);
  g_wait_limit_ns.store(wait_limit_ns);
  return SDPA_OK;
}
