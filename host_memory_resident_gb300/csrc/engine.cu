// Streaming engine and C ABI of the training step.
//
// The step follows the RAM-centric method of the MegaTrain articles:
//  * host-resident state: FP32 master / m / v / grad in caller memory, a
//    pinned bf16 flat store of all weights ("layer_pinned_flats", lqnn.cn
//    article section 三.1) that the host Adam rewrites per unit;
//  * two fixed device flat buffers ("gpu_flat_buffers", same section) that
//    units (embedding, each layer, final norm + head) are copied into on a
//    host-to-device stream; the compute stream waits a weight_ready event
//    and records buffer_free when done, the copy stream waits buffer_free
//    before overwriting (section 三.2: three streams, weight_ready_events /
//    buffer_free_events; zhichai.net article point 2, ping-pong buffers);
//  * checkpoint recompute: the input of every C-th layer is kept, backward
//    walks segments from last to first and recomputes each from its
//    checkpoint (section 三.4; zhichai.net article point 3), except the last
//    segment, whose activations the forward leaves in place;
//  * a K-slab device gradient pool: a unit's weight gradients land in a free
//    slab, a device-to-host stream copies it to pinned staging, and a host
//    worker thread adds it into the FP32 gradient and runs Adam on that unit
//    (section 三.3, "GPU backward -> gradient DMA -> CPU accumulate").
// Everything on the device is the library's own kernels; there is no CPU
// fallback for the layer compute.
#include <omp.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <condition_variable>
#include <cstdio>
#include <cstring>
#include <deque>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "common.cuh"
#include "host_math.h"
#include "mt_internal.h"

namespace mt {
namespace {

thread_local std::string g_thread_error;
std::atomic<int> g_fail_next_alloc{0};

using Clock = std::chrono::steady_clock;

double seconds_since(Clock::time_point t0) {
  return std::chrono::duration<double>(Clock::now() - t0).count();
}

struct StepError {
  int code;
  std::string msg;
};

#define CK(call)                                                                                     \
  do {                                                                                               \
    cudaError_t e_ = (call);                                                                         \
    if (e_ != cudaSuccess) throw StepError{MT_ECUDA, std::string(#call ": ") + cudaGetErrorString(e_)}; \
  } while (0)

#define KK(call)                                                                      \
  do {                                                                                \
    int r_ = (call);                                                                  \
    if (r_ != MT_OK) throw StepError{r_, std::string("kernel launch failed: ") + #call}; \
  } while (0)

// Device arena: one allocation carved into 256-byte aligned pieces.
struct Arena {
  uint8_t* base = nullptr;
  size_t cap = 0, used = 0;
  void* take(size_t bytes) {
    size_t off = (used + 255) & ~size_t(255);
    if (off + bytes > cap) throw StepError{MT_ENOMEM, "device arena exhausted"};
    used = off + bytes;
    return base + off;
  }
};

template <typename T>
T* take(Arena& a, size_t n) {
  return reinterpret_cast<T*>(a.take(sizeof(T) * (n ? n : 1)));
}

// Activations saved for one layer's backward. The residual stream (layer
// input x, h, the checkpoints) is fp32: the method's bf16 storage is that of
// the weights, gradients and the operands of the products, and the stream
// itself is no operand (rounding it to bf16 twice per layer compounds with
// depth).
struct Saved {
  float* x;    // layer input [M, d] (fp32 residual stream)
  bf16* u;     // attention-norm output [M, d]
  float* r1;   // its rstd [M]
  bf16* qkv;   // q, k (after RoPE), v [M, qkvN]
  bf16* o;     // attention output [M, hq]
  float* lse;  // [B, H, s]
  float* h;    // after attention residual [M, d] (fp32)
  bf16* z;     // mlp-norm output [M, d]
  float* r2;   // [M]
  bf16* gu;    // gate | up [M, 2f]
  bf16* a;     // silu(g) * u [M, f]
};

struct Job {
  int unit;
  int slab;
  int64_t t;
  int parity;     // step parity: selects the step's loss event / state
  int64_t seq;    // step sequence number (monotonic per handle)
  bool acc;       // add to the running gradient sum (micro-steps after the first)
  bool adam;      // last micro-step: apply Adam to (sum) * scale
  float scale;
  std::chrono::steady_clock::time_point step0;  // host time the step began (timeline)
};

}  // namespace
}  // namespace mt

struct mt_handle {
  mt_config cfg;
  mt::FlatLayout lay;
  float *master, *adam_m, *adam_v, *grad;
  int64_t n_total;
  int threads;
  int64_t t = 0;  // Adam steps taken
  int broken = 0;
  std::string err;

  // dims
  int L, d, H, Hkv, hd, f, V, qkvN, hq, nseg, Mmax, Mchunk;

  // host memory (pinned)
  uint16_t* store = nullptr;
  std::vector<uint16_t*> staging;
  int32_t* tok_pinned = nullptr;  // tokens | labels
  float* loss_pinned = nullptr;
  int32_t* flag_pinned = nullptr;

  // device memory
  void* dmem = nullptr;
  size_t dbytes = 0;
  mt::bf16* wbuf[2] = {nullptr, nullptr};
  mt::bf16* resident = nullptr;
  std::vector<mt::bf16*> slab;
  int32_t *d_tok = nullptr, *d_lab = nullptr, *d_flag = nullptr, *d_ework = nullptr;
  float *cos_t = nullptr, *sin_t = nullptr;
  float *xa = nullptr, *xb = nullptr;   // fp32 residual stream between checkpoints
  std::vector<float*> ckpt;             // fp32 layer inputs, one per segment
  std::vector<mt::Saved> saved;
  // keep_attention: every layer's attention output and log-sum-exp from the
  // forward, so the backward's recompute skips the attention core
  std::vector<mt::bf16*> att_o;
  std::vector<float*> att_lse;
  mt::bf16 *xh = nullptr, *dz = nullptr;
  float *rf = nullptr, *logits = nullptr, *loss_rows = nullptr, *loss_dev = nullptr;
  float *dx32 = nullptr, *dh32 = nullptr, *dn32 = nullptr, *delta = nullptr, *npart = nullptr;
  mt::bf16 *dxb = nullptr, *dhb = nullptr, *da = nullptr, *dob = nullptr, *dqkv = nullptr;
  // head: dz per chunk of Mchunk rows (dz_chunked) with the head's weight
  // gradient summed in fp32 (dhead32, V x d), else dz for every token
  bool dz_chunked = false;
  float* dhead32 = nullptr;
  // fp32 partial products of the weight gradients that are split along K
  float* wg_ws = nullptr;
  size_t wg_ws_elems = 0;

  // streams and events
  cudaStream_t s_comp = nullptr, s_h2d = nullptr, s_d2h = nullptr;
  cudaEvent_t ev_ready[2] = {nullptr, nullptr}, ev_free[2] = {nullptr, nullptr};
  std::vector<cudaEvent_t> ev_slab_ready, ev_d2h_done;
  cudaEvent_t ev_loss[2] = {nullptr, nullptr}, ev_resident = nullptr;
  int slot_unit[2] = {-1, -1};
  int slot_last_use[2] = {0, 0};
  int use_clock = 0;
  int next_slab = 0;

  // worker
  std::thread worker;
  std::mutex mu;
  std::condition_variable cv;
  std::deque<mt::Job> jobs;
  std::vector<int> staging_busy;
  int units_done = 0;
  int in_flight = 0;
  bool stop = false;
  int worker_error = 0;
  std::string worker_msg;
  int loss_state[2] = {0, 0};  // per step parity: 0 unknown, 1 finite, 2 non-finite
  std::vector<int> unit_pending;  // queued or running jobs per unit
  int64_t step_seq = 0;        // sequence number of the step being enqueued
  bool accum_nonfinite = false;  // a micro-step of the current accumulation had a non-finite loss
  int64_t inject_sleep_ms = 0, inject_fail_at = 0, deadline_ms = 600000;
  int64_t worker_units_total = 0;

  // stats and the optional per-kernel profile (CUDA events on the compute stream)
  mt_stats st{};
  int prof_on = 0;
  std::vector<cudaEvent_t> prof_events;
  struct ProfRec { int cat, stream; double flops, bytes; };
  std::vector<ProfRec> prof_recs;
  mt_kernel_profile prof{};
  cudaEvent_t prof_ref = nullptr;        // start of the last profiled step (compute stream)
  std::vector<mt_timeline_rec> timeline;  // its launches and copies
  int64_t timeline_seq = -1;             // that step's sequence number
  std::vector<mt_timeline_rec> host_tl;   // worker records of step host_tl_seq (under mu)
  int64_t host_tl_seq = -1;
  std::chrono::steady_clock::time_point host_tl_step0{};
  // the step before: its records, relative to its own start
  std::vector<mt_timeline_rec> host_tl_prev;
  int64_t host_tl_prev_seq = -1;
  std::chrono::steady_clock::time_point host_tl_prev_step0{};
  std::chrono::steady_clock::time_point step0{};  // host time the current step began
};

namespace mt {
namespace {
// The down projection's input gradient takes the SwiGLU backward in its
// epilogue (so the da buffer is not needed) unless the configuration asks
// for the separate kernels or the ffn width does not fit the fused form.
bool swiglu_bwd_fused(const mt_handle* h) { return !h->cfg.unfused_epilogues && h->f % 32 == 0; }


void set_err(mt_handle* h, const std::string& m) {
  if (h) h->err = m;
  g_thread_error = m;
}

// ------------------------------------------------------------------ worker
void worker_main(mt_handle* h) {
  for (;;) {
    Job job;
    {
      std::unique_lock<std::mutex> lk(h->mu);
      h->cv.wait(lk, [&] { return h->stop || !h->jobs.empty(); });
      if (h->stop && h->jobs.empty()) return;
      // Order: older steps first, then the lowest unit among jobs whose slab
      // copy has landed. The next step's forward needs units lowest first,
      // so the units it needs last (the top layers, whose gradients land
      // first) are left for the end of the pass and the forward starts
      // while the worker is still busy; a unit that lands while others wait
      // is taken ahead of them. The worker never idles on one copy while
      // other slabs are ready. At most K jobs are queued: the scan and its
      // non-blocking event queries are cheap.
      // When no copy has landed, the earliest issued one (the queue is in
      // issue order) is the one to wait for.
      auto it = h->jobs.end();
      for (auto j = h->jobs.begin(); j != h->jobs.end(); ++j) {
        if (cudaEventQuery(h->ev_d2h_done[j->slab]) != cudaSuccess) continue;
        if (it == h->jobs.end() || j->seq < it->seq || (j->seq == it->seq && j->unit < it->unit)) it = j;
      }
      if (it == h->jobs.end()) it = h->jobs.begin();
      job = *it;
      h->jobs.erase(it);
      h->in_flight = 1;
    }
    int code = MT_OK;
    std::string msg;
    double wait_s = 0.0, compute_s = 0.0;
    const auto t0 = Clock::now();
    const auto deadline = t0 + std::chrono::milliseconds(h->deadline_ms);
    if (h->inject_sleep_ms > 0) std::this_thread::sleep_for(std::chrono::milliseconds(h->inject_sleep_ms));
    ++h->worker_units_total;
    if (h->inject_fail_at > 0 && h->worker_units_total == h->inject_fail_at) {
      code = MT_EWORKER;
      msg = "injected worker failure";
    }
    // wait for the slab copy (and, once per step, the loss) to land
    auto wait_event = [&](cudaEvent_t ev) -> bool {
      for (;;) {
        cudaError_t q = cudaEventQuery(ev);
        if (q == cudaSuccess) return true;
        if (q != cudaErrorNotReady) {
          code = MT_ECUDA;
          msg = std::string("worker event query: ") + cudaGetErrorString(q);
          return false;
        }
        if (Clock::now() > deadline) {
          code = MT_ETIMEOUT;
          msg = "worker timed out waiting for a device-to-host copy";
          return false;
        }
        std::this_thread::sleep_for(std::chrono::microseconds(20));
      }
    };
    const auto tw = Clock::now();
    if (code == MT_OK && wait_event(h->ev_d2h_done[job.slab]) && h->loss_state[job.parity] == 0 &&
        wait_event(h->ev_loss[job.parity])) {
      const float total = h->loss_pinned[job.parity];
      h->loss_state[job.parity] = std::isfinite(total) ? 1 : 2;
    }
    if (code == MT_OK) {
      AdamArgs a;
      const int64_t off = h->lay.unit_off[job.unit];
      a.w = h->master + off;
      a.m = h->adam_m + off;
      a.v = h->adam_v + off;
      a.grad_out = h->grad ? h->grad + off : nullptr;
      a.grad_in = nullptr;
      a.slab = h->staging[job.slab];
      a.store = h->store + off;
      a.n = h->lay.unit_len[job.unit];
      a.t = job.t;
      a.lr = h->cfg.lr;
      a.beta1 = h->cfg.beta1;
      a.beta2 = h->cfg.beta2;
      a.eps = h->cfg.adam_eps;
      a.apply = job.adam && h->loss_state[job.parity] == 1 && !h->accum_nonfinite;
      a.accumulate = job.acc;
      a.grad_scale = job.scale;
      const auto tc = Clock::now();
      wait_s = std::chrono::duration<double>(tc - tw).count();
      adam_pass(a, h->threads);
      compute_s = seconds_since(tc);
      if (h->prof_on) {
        auto ms = [&](Clock::time_point x) { return std::chrono::duration<double, std::milli>(x - job.step0).count(); };
        const double t_end = ms(Clock::now());
        std::lock_guard<std::mutex> lk(h->mu);
        if (job.seq != h->host_tl_seq) {
          h->host_tl_prev.swap(h->host_tl);
          h->host_tl_prev_seq = h->host_tl_seq;
          h->host_tl_prev_step0 = h->host_tl_step0;
          h->host_tl.clear();
          h->host_tl_seq = job.seq;
          h->host_tl_step0 = job.step0;
        }
        h->host_tl.push_back(mt_timeline_rec{job.unit, 4, ms(tw), ms(tc)});
        h->host_tl.push_back(mt_timeline_rec{job.unit, 3, ms(tc), t_end});
      }
    }
    {
      std::lock_guard<std::mutex> lk(h->mu);
      h->st.host_adam_s += seconds_since(t0);
      h->st.host_compute_s += compute_s;
      h->st.host_copy_wait_s += wait_s;
      h->staging_busy[job.slab] = 0;
      h->in_flight = 0;
      --h->unit_pending[job.unit];
      ++h->units_done;
      if (code != MT_OK && h->worker_error == 0) {
        h->worker_error = code;
        h->worker_msg = msg;
      }
    }
    h->cv.notify_all();
  }
}

// ------------------------------------------------------------ the step
struct Step {
  mt_handle* h;
  int B, s, M;
  int64_t t_next;
  bool acc = false, adam = true;
  float gscale = 1.f;

  cudaStream_t cs() const { return h->s_comp; }

  // Make unit `u`'s weights usable on the compute stream; returns its base.
  int parity() const { return (int)(t_next & 1); }

  // With overlap, a unit's bf16 store may still be rewritten by the previous
  // step's Adam: wait (on the host, before its upload is enqueued) until the
  // worker has no job left for it.
  void wait_unit_updated(int u) {
    if (!h->cfg.overlap_adam) return;
    const auto t0 = Clock::now();
    std::unique_lock<std::mutex> lk(h->mu);
    const bool ok = h->cv.wait_for(lk, std::chrono::milliseconds(h->deadline_ms),
                                   [&] { return h->unit_pending[u] == 0 || h->worker_error; });
    h->st.host_wait_s += seconds_since(t0);
    if (h->worker_error) throw StepError{h->worker_error, h->worker_msg};
    if (!ok) throw StepError{MT_ETIMEOUT, "timed out waiting for a unit's host optimizer update"};
  }

  bf16* acquire(int u) {
    if (!h->cfg.streamed) return h->resident + h->lay.unit_off[u];
    int slot = -1;
    for (int i = 0; i < 2; ++i)
      if (h->slot_unit[i] == u) slot = i;
    if (slot < 0) {
      wait_unit_updated(u);
      slot = h->slot_last_use[0] <= h->slot_last_use[1] ? 0 : 1;
      const size_t bytes = sizeof(uint16_t) * h->lay.unit_len[u];
      CK(cudaStreamWaitEvent(h->s_h2d, h->ev_free[slot], 0));
      prof_copy_begin(h->s_h2d);
      CK(cudaMemcpyAsync(h->wbuf[slot], h->store + h->lay.unit_off[u], bytes, cudaMemcpyHostToDevice, h->s_h2d));
      prof_copy_end(h->s_h2d, MT_PROF_H2D, (double)bytes);
      CK(cudaEventRecord(h->ev_ready[slot], h->s_h2d));
      h->slot_unit[slot] = u;
      h->st.h2d_bytes += (int64_t)bytes;
      h->st.h2d_units += 1;
    }
    h->slot_last_use[slot] = ++h->use_clock;
    CK(cudaStreamWaitEvent(h->s_comp, h->ev_ready[slot], 0));
    cur_slot = slot;
    return h->wbuf[slot];
  }
  int cur_slot = -1;
  void release() {
    if (h->cfg.streamed && cur_slot >= 0) CK(cudaEventRecord(h->ev_free[cur_slot], h->s_comp));
    cur_slot = -1;
  }

  // Take a slab for a unit's weight gradients: any whose host staging the
  // worker has consumed (the worker takes units out of arrival order, so
  // slabs come free out of order too). Blocks, with the deadline, while all
  // K are held: the back-pressure that keeps the backward at most K units
  // ahead of the host.
  int slab_begin() {
    const int n = h->cfg.n_slabs;
    int k = -1;
    const auto t0 = Clock::now();
    {
      std::unique_lock<std::mutex> lk(h->mu);
      auto pick = [&] {
        for (int i = 0; i < n; ++i) {
          const int j = (h->next_slab + i) % n;
          if (!h->staging_busy[j]) {
            k = j;
            return true;
          }
        }
        return false;
      };
      const bool ok = h->cv.wait_for(lk, std::chrono::milliseconds(h->deadline_ms),
                                     [&] { return h->worker_error || pick(); });
      h->st.host_wait_s += seconds_since(t0);
      if (h->worker_error) throw StepError{h->worker_error, h->worker_msg};
      if (!ok) throw StepError{MT_ETIMEOUT, "timed out waiting for a free gradient slab"};
      h->staging_busy[k] = 1;
      h->next_slab = (k + 1) % n;
    }
    // the slab's previous copy has landed (the worker consumed it); the wait
    // orders the device-side reuse after it
    CK(cudaStreamWaitEvent(h->s_comp, h->ev_d2h_done[k], 0));
    return k;
  }
  // Ship slab k of unit u to the host and queue it for the worker.
  void slab_end(int k, int u) {
    CK(cudaEventRecord(h->ev_slab_ready[k], h->s_comp));
    const size_t bytes = sizeof(uint16_t) * h->lay.unit_len[u];
    CK(cudaStreamWaitEvent(h->s_d2h, h->ev_slab_ready[k], 0));
    prof_copy_begin(h->s_d2h);
    CK(cudaMemcpyAsync(h->staging[k], h->slab[k], bytes, cudaMemcpyDeviceToHost, h->s_d2h));
    prof_copy_end(h->s_d2h, MT_PROF_D2H, (double)bytes);
    CK(cudaEventRecord(h->ev_d2h_done[k], h->s_d2h));
    h->st.d2h_bytes += (int64_t)bytes;
    {
      std::lock_guard<std::mutex> lk(h->mu);
      h->jobs.push_back(Job{u, k, t_next, parity(), h->step_seq, acc, adam, gscale, h->step0});
      ++h->unit_pending[u];
    }
    h->cv.notify_all();
  }

  // Kernel launch bookkeeping: count launches and, when profiling is on,
  // bracket the launch with a pair of events on the compute stream.
  size_t prof_next = 0;
  void prof_begin() {
    if (!h->prof_on) return;
    while (h->prof_events.size() < 2 * (prof_next + 1)) {
      cudaEvent_t e;
      CK(cudaEventCreate(&e));
      h->prof_events.push_back(e);
    }
    CK(cudaEventRecord(h->prof_events[2 * prof_next], cs()));
  }
  void prof_end(int cat, int launches, double flops, double bytes) {
    h->st.kernel_launches += launches;
    h->prof.launches[cat] += launches;
    if (!h->prof_on) return;
    CK(cudaEventRecord(h->prof_events[2 * prof_next + 1], cs()));
    h->prof_recs.push_back({cat, 0, flops, bytes});
    ++prof_next;
  }
  // A copy on `st`, bracketed by events on that stream when profiling is on.
  void prof_copy_begin(cudaStream_t st) {
    if (!h->prof_on) return;
    while (h->prof_events.size() < 2 * (prof_next + 1)) {
      cudaEvent_t e;
      CK(cudaEventCreate(&e));
      h->prof_events.push_back(e);
    }
    CK(cudaEventRecord(h->prof_events[2 * prof_next], st));
  }
  void prof_copy_end(cudaStream_t st, int cat, double bytes) {
    h->prof.launches[cat] += 1;
    if (!h->prof_on) return;
    CK(cudaEventRecord(h->prof_events[2 * prof_next + 1], st));
    h->prof_recs.push_back({cat, st == h->s_h2d ? 1 : 2, 0.0, bytes});
    ++prof_next;
  }
#define KP(cat, nl, fl, by, call) \
  do {                            \
    prof_begin();                 \
    KK(call);                     \
    prof_end(cat, nl, fl, by);    \
  } while (0)

  // C[M,N] = A[M,K] * B[N,K]^T (+R)
  void gemm(const bf16* A, long long lda, const bf16* Bm, long long ldb, void* C, long long ldc, bool f32,
            const void* R, long long ldr, int m, int n, int k) {
    const double bytes = 2.0 * ((double)m * k + (double)n * k) + (f32 ? 4.0 : 2.0) * m * n * (R ? 2.0 : 1.0);
    KP(MT_PROF_GEMM, 1, 2.0 * m * n * k, bytes,
       gemm_abt(A, lda, Bm, ldb, C, ldc, f32 ? 1 : 0, R, ldr, m, n, k, cs()));
  }
  // C[M,N] = op(A) * op(B)^T (+R) with A and/or B read MN-major in place
  void gemm_mn(const bf16* A, long long lda, bool a_mn, const bf16* Bm, long long ldb, bool b_mn, void* C,
               long long ldc, bool f32, int m, int n, int k) {
    const double bytes = 2.0 * ((double)m * k + (double)n * k) + (f32 ? 4.0 : 2.0) * m * n;
    KP(MT_PROF_GEMM, 1, 2.0 * m * n * k, bytes,
       gemm_ex(A, lda, a_mn ? 1 : 0, Bm, ldb, b_mn ? 1 : 0, C, ldc, f32 ? 1 : 0, nullptr, 0, m, n, k, cs()));
  }
  // Weight gradient g[m, n] = dY^T X over the step's M tokens (both read
  // token-major), split along the tokens when the output has few tiles.
  void gemm_wg(const bf16* dY, long long ldy, const bf16* X, long long ldx, bf16* g, long long ldg, int m, int n) {
    const int sp = splitk_factor(m, n, M);
    const double bytes = 2.0 * ((double)m * M + (double)n * M) + 2.0 * m * n;
    KP(MT_PROF_GEMM, sp > 1 ? 2 : 1, 2.0 * m * n * (double)M, bytes,
       gemm_wgrad(dY, ldy, 1, X, ldx, 1, g, ldg, m, n, M, h->wg_ws, h->wg_ws_elems, cs()));
  }
  double attn_flops(bool bwd) const {
    // causal: half of the s x s score matrix; forward 2 products, backward 5
    const double per = 2.0 * B * (double)h->H * s * (double)s * h->hd / 2.0;
    return (bwd ? 5.0 : 2.0) * per;
  }
  // fp32 x in, bf16 y out (+ rstd); backward: fp32 dy and x in, fp32 and
  // bf16 dx out (+ the fp32 residual-branch gradient in)
  double norm_fwd_bytes() const { return 6.0 * M * h->d + 4.0 * M; }
  double norm_bwd_bytes(bool res) const { return (4.0 + 4.0 + 4.0 + 2.0 + (res ? 4.0 : 0.0)) * M * h->d; }
  double rope_bytes() const { return 4.0 * M * (h->H + h->Hkv) * h->hd; }
  // RoPE and SwiGLU go into the GEMM epilogues unless the configuration asks
  // for the separate kernels or a shape does not fit the fused forms.
  bool fuse_rope() const { return !h->cfg.unfused_epilogues && h->hd % 64 == 0 && 128 % h->hd == 0; }
  bool fuse_swiglu_fwd() const { return !h->cfg.unfused_epilogues && h->f % 128 == 0; }
  bool fuse_swiglu_bwd() const { return swiglu_bwd_fused(h); }

  // Forward of layer l with weights W; writes the saved activations into S and
  // the layer output into x_out.
  // With keep_attention, S.o / S.lse point at layer l's kept tensors; the
  // forward writes them and a recompute reads them instead of re-running the
  // attention (the same values, so the step's results are unchanged).
  void layer_fwd(const bf16* W, const Saved& S, float* x_out, bool recompute = false) {
    const LayerOffsets& o = h->lay.layer;
    const int d = h->d, f = h->f;
    KP(MT_PROF_NORM, 1, 0.0, norm_fwd_bytes(),
       mt_k_rmsnorm_fwd(S.x, 1, W + o.attn_norm, S.u, S.r1, M, d, h->cfg.rms_eps, cs()));
    if (fuse_rope()) {
      const int qn = h->qkvN;
      const double bytes = 2.0 * ((double)M * d + (double)qn * d + (double)M * qn) + 8.0 * s * (h->hd / 2);
      KP(MT_PROF_GEMM, 1, 2.0 * M * (double)qn * d, bytes,
         gemm_rope(S.u, d, W + o.wqkv, d, S.qkv, qn, M, qn, d, h->cos_t, h->sin_t, (h->H + h->Hkv) * h->hd, h->hd,
                   s, cs()));
    } else {
      gemm(S.u, d, W + o.wqkv, d, S.qkv, h->qkvN, false, nullptr, 0, M, h->qkvN, d);
      KP(MT_PROF_ROPE, 1, 0.0, rope_bytes(),
         mt_k_rope(S.qkv, h->qkvN, B, s, h->H + h->Hkv, h->hd, h->cos_t, h->sin_t, 0, cs()));
    }
    if (!(recompute && h->cfg.keep_attention))
      KP(MT_PROF_ATTN_FWD, 1, attn_flops(false), 0.0,
         mt_k_attn_fwd(S.qkv, h->qkvN, S.o, h->hq, S.lse, B, s, h->H, h->Hkv, h->hd, cs()));
    // h = x + o Wo^T and x_out = h + a Wdown^T stay fp32
    gemm(S.o, h->hq, W + o.wo, h->hq, S.h, d, true, S.x, d, M, d, h->hq);
    KP(MT_PROF_NORM, 1, 0.0, norm_fwd_bytes(),
       mt_k_rmsnorm_fwd(S.h, 1, W + o.mlp_norm, S.z, S.r2, M, d, h->cfg.rms_eps, cs()));
    if (fuse_swiglu_fwd()) {
      const double bytes = 2.0 * ((double)M * d + 2.0 * f * d + 2.0 * M * f + (double)M * f);
      KP(MT_PROF_GEMM, 1, 2.0 * M * (2.0 * f) * d, bytes,
         gemm_swiglu_fwd(S.z, d, W + o.wgu, d, S.gu, 2 * f, S.a, f, M, f, d, cs()));
    } else {
      gemm(S.z, d, W + o.wgu, d, S.gu, 2 * f, false, nullptr, 0, M, 2 * f, d);
      KP(MT_PROF_SWIGLU, 1, 0.0, 6.0 * M * f, mt_k_swiglu_fwd(S.gu, S.a, M, f, cs()));
    }
    gemm(S.a, f, W + o.wdown, f, x_out, d, true, S.h, d, M, d, f);
  }

  // Backward of one layer: reads dx32/dxb (gradient w.r.t. the layer output),
  // writes the gradient w.r.t. its input back into dx32/dxb and the weight
  // gradients into slab `g`.
  void layer_bwd(const bf16* W, const Saved& S, bf16* g) {
    const LayerOffsets& o = h->lay.layer;
    const int d = h->d, f = h->f, hq = h->hq, qn = h->qkvN;
    // Weight gradients dW = dY^T X read both token-major activations in place
    // (MN-major operands, K = tokens); input gradients dX = dY W read the
    // weight [out, in] in place as a [K, N] operand. Nothing is transposed.
    // down projection: dWdown = dy^T a ; da = dy Wdown. d(gate | up)
    // overwrites the saved gate | up in place (each element is read before it
    // is written, by the same thread; nothing reads gate | up afterwards)
    bf16* dgu = S.gu;
    gemm_wg(h->dxb, d, S.a, f, g + o.wdown, f, d, f);
    if (fuse_swiglu_bwd()) {
      // da = dy Wdown stays in the SM; the epilogue writes d(gate) | d(up)
      const double bytes = 2.0 * ((double)M * d + (double)d * f + 2.0 * M * f + 2.0 * M * f);
      KP(MT_PROF_GEMM, 1, 2.0 * M * (double)f * d, bytes,
         gemm_swiglu_bwd(h->dxb, d, W + o.wdown, f, S.gu, 2 * f, dgu, 2 * f, M, f, d, cs()));
    } else {
      gemm_mn(h->dxb, d, false, W + o.wdown, f, true, h->da, f, false, M, f, d);
      KP(MT_PROF_SWIGLU, 1, 0.0, 10.0 * M * f, mt_k_swiglu_bwd(h->da, S.gu, dgu, M, f, cs()));
    }
    // gate/up projection
    gemm_wg(dgu, 2 * f, S.z, d, g + o.wgu, d, 2 * f, d);
    gemm_mn(dgu, 2 * f, false, W + o.wgu, d, true, h->dn32, d, true, M, d, 2 * f);
    KP(MT_PROF_NORM, 2, 0.0, norm_bwd_bytes(true),
       mt_k_rmsnorm_bwd(h->dn32, S.h, 1, W + o.mlp_norm, S.r2, h->dx32, h->dh32, h->dhb, h->npart, g + o.mlp_norm, M,
                        d, cs()));
    // output projection
    gemm_wg(h->dhb, d, S.o, hq, g + o.wo, hq, d, hq);
    gemm_mn(h->dhb, d, false, W + o.wo, hq, true, h->dob, hq, false, M, hq, d);
    // attention, and RoPE's inverse rotation of dq / dk (in the tcgen05
    // kernels' stores at hd 64 / 128; a separate pass at hd 16)
    const bool tc_attn = h->hd == 64 || h->hd == 128;
    KP(MT_PROF_ATTN_BWD, tc_attn ? 3 : 4, attn_flops(true), 0.0,
       mt_k_attn_bwd_rope(S.qkv, qn, S.o, hq, h->dob, hq, S.lse, h->delta, h->dqkv, qn, B, s, h->H, h->Hkv, h->hd,
                          h->cos_t, h->sin_t, cs()));
    // qkv projection
    gemm_wg(h->dqkv, qn, S.u, d, g + o.wqkv, d, qn, d);
    gemm_mn(h->dqkv, qn, false, W + o.wqkv, d, true, h->dn32, d, true, M, d, qn);
    KP(MT_PROF_NORM, 2, 0.0, norm_bwd_bytes(true),
       mt_k_rmsnorm_bwd(h->dn32, S.x, 1, W + o.attn_norm, S.r1, h->dh32, h->dx32, h->dxb, h->npart, g + o.attn_norm, M,
                        d, cs()));
  }

  // Final norm, logits, cross entropy and their backward (head unit). The
  // logits are made Mchunk rows at a time (fp32). dz is kept for every token
  // and the head's two gradient products run once over all of them, or, when
  // the handle keeps dz per chunk (dz_chunked), each chunk's products run
  // right after its cross entropy: dxh rows of the chunk, and the head's
  // weight gradient summed over the chunks in an fp32 accumulator that is
  // rounded to bf16 once at the end.
  void head(const bf16* W, const float* xL, bf16* g) {
    const int d = h->d, V = h->V;
    const bf16* wf = W + h->lay.final_norm;
    const bf16* head = W + h->lay.head;
    KP(MT_PROF_NORM, 1, 0.0, norm_fwd_bytes(), mt_k_rmsnorm_fwd(xL, 1, wf, h->xh, h->rf, M, d, h->cfg.rms_eps, cs()));
    const float scale = 1.f / (float)M;
    const bool per_chunk = h->dz_chunked && M > h->Mchunk;
    for (int r0 = 0; r0 < M; r0 += h->Mchunk) {
      const int mc = std::min(h->Mchunk, M - r0);
      bf16* dzc = per_chunk ? h->dz : h->dz + (size_t)r0 * V;
      gemm(h->xh + (size_t)r0 * d, d, head, d, h->logits, V, true, nullptr, 0, mc, V, d);
      KP(MT_PROF_CE, 1, 0.0, 6.0 * mc * (double)V,
         mt_k_cross_entropy(h->logits, V, h->d_lab + r0, dzc, V, h->loss_rows + r0, mc, V, scale, cs()));
      if (per_chunk) {
        // dxh of the chunk's rows = dz_c Head; dHead (+)= dz_c^T xh_c
        gemm_mn(dzc, V, false, head, d, true, h->dn32 + (size_t)r0 * d, d, true, mc, d, V);
        const double bytes = 2.0 * ((double)mc * V + (double)mc * d) + 4.0 * V * (double)d * (r0 > 0 ? 2.0 : 1.0);
        KP(MT_PROF_GEMM, 1, 2.0 * V * (double)d * mc, bytes,
           gemm_ex(dzc, V, 1, h->xh + (size_t)r0 * d, d, 1, h->dhead32, d, 1, r0 > 0 ? h->dhead32 : nullptr, d, V,
                   d, mc, cs()));
      }
    }
    KP(MT_PROF_OTHER, 1, 0.0, 4.0 * M, mt_k_sum(h->loss_rows, M, h->loss_dev, cs()));
    CK(cudaMemcpyAsync(h->loss_pinned + parity(), h->loss_dev, sizeof(float), cudaMemcpyDeviceToHost, cs()));
    CK(cudaEventRecord(h->ev_loss[parity()], cs()));
    if (per_chunk) {
      KP(MT_PROF_OTHER, 1, 0.0, 6.0 * V * (double)d,
         convert_f32_bf16(h->dhead32, g + h->lay.head, (long long)V * d, cs()));
    } else {
      // dHead = dz^T xh ; dxh = dz Head (both read in place)
      gemm_wg(h->dz, V, h->xh, d, g + h->lay.head, d, V, d);
      gemm_mn(h->dz, V, false, head, d, true, h->dn32, d, true, M, d, V);
    }
    KP(MT_PROF_NORM, 2, 0.0, norm_bwd_bytes(false),
       mt_k_rmsnorm_bwd(h->dn32, xL, 1, wf, h->rf, nullptr, h->dx32, h->dxb, h->npart, g + h->lay.final_norm, M, d,
                        cs()));
  }

  void run() {
    mt_handle& hh = *h;
    const int L = hh.L, C = hh.cfg.ckpt_interval;
    {
      // the state of this parity belongs to the step before last, whose
      // units were all updated before the previous forward could use them
      std::lock_guard<std::mutex> lk(hh.mu);
      hh.loss_state[parity()] = 0;
      ++hh.step_seq;
    }
    hh.step0 = Clock::now();
    if (hh.prof_on) {
      if (!hh.prof_ref) CK(cudaEventCreate(&hh.prof_ref));
      CK(cudaEventRecord(hh.prof_ref, hh.s_comp));
    }
    // The host Adam rewrote the bf16 store since the last step, so nothing
    // left in the two device buffers may be reused: forget their contents.
    hh.slot_unit[0] = hh.slot_unit[1] = -1;
    if (!hh.cfg.streamed) {
      for (int u = 0; u < L + 2; ++u) wait_unit_updated(u);
      const size_t bytes = sizeof(uint16_t) * hh.n_total;
      CK(cudaMemcpyAsync(hh.resident, hh.store, bytes, cudaMemcpyHostToDevice, hh.s_h2d));
      CK(cudaEventRecord(hh.ev_resident, hh.s_h2d));
      CK(cudaStreamWaitEvent(hh.s_comp, hh.ev_resident, 0));
      hh.st.h2d_bytes += (int64_t)bytes;
      hh.st.h2d_units += L + 2;
    }
    // ---- forward: embedding, layers (checkpoint every C), head
    {
      bf16* E = acquire(0);
      KP(MT_PROF_EMBED, 1, 0.0, 4.0 * M * hh.d,
         mt_k_embedding_fwd(E + (hh.lay.embed - hh.lay.unit_off[0]), hh.d_tok, hh.ckpt[0], 1, M, hh.d, hh.V, cs()));
      release();
    }
    // The last segment's layers keep their activations in the saved sets,
    // exactly where its recompute would put them, so the backward starts on
    // that segment without recomputing it.
    const int last_a = (hh.nseg - 1) * C;
    float* x = hh.ckpt[0];
    for (int l = 0; l < L; ++l) {
      bf16* W = acquire(1 + l);
      float* out;
      if (l >= last_a) {
        Saved& S = hh.saved[l - last_a];
        if (l == last_a) S.x = hh.ckpt[hh.nseg - 1];
        if (hh.cfg.keep_attention) {
          S.o = hh.att_o[l];
          S.lse = hh.att_lse[l];
        }
        out = (l + 1 < L) ? hh.saved[l + 1 - last_a].x : hh.xa;
        layer_fwd(W, S, out);
      } else {
        Saved S = hh.saved[0];
        S.x = x;
        if (hh.cfg.keep_attention) {
          S.o = hh.att_o[l];
          S.lse = hh.att_lse[l];
        }
        if ((l + 1) % C == 0) out = hh.ckpt[(l + 1) / C];
        else out = (x == hh.xa) ? hh.xb : hh.xa;
        layer_fwd(W, S, out);
      }
      release();
      x = out;
    }
    {
      bf16* W = acquire(L + 1);
      const int k = slab_begin();
      head(W, x, hh.slab[k]);
      release();
      slab_end(k, L + 1);
    }
    // ---- backward over segments, last to first, recomputing all but the last
    for (int seg = hh.nseg - 1; seg >= 0; --seg) {
      const int a = seg * C, b = std::min(L, a + C);
      for (int l = a; l < b && seg < hh.nseg - 1; ++l) {
        bf16* W = acquire(1 + l);
        Saved& S = hh.saved[l - a];
        if (l == a) S.x = hh.ckpt[seg];
        if (hh.cfg.keep_attention) {
          S.o = hh.att_o[l];
          S.lse = hh.att_lse[l];
        }
        float* out = (l + 1 < b) ? hh.saved[l + 1 - a].x : hh.xa;
        layer_fwd(W, S, out, true);
        release();
      }
      for (int l = b - 1; l >= a; --l) {
        bf16* W = acquire(1 + l);
        const int k = slab_begin();
        layer_bwd(W, hh.saved[l - a], hh.slab[k]);
        release();
        slab_end(k, 1 + l);
      }
    }
    {
      const int k = slab_begin();
      KP(MT_PROF_EMBED, 2, 0.0, 4.0 * M * hh.d + 2.0 * hh.V * (double)hh.d,
         mt_k_embedding_bwd(hh.dx32, hh.d_tok, hh.slab[k] + 0, M, hh.d, hh.V, hh.d_ework, cs()));
      slab_end(k, 0);
    }
  }
};

void destroy_resources(mt_handle* h) {
  if (h->worker.joinable()) {
    {
      std::lock_guard<std::mutex> lk(h->mu);
      h->stop = true;
    }
    h->cv.notify_all();
    h->worker.join();
  }
  if (h->s_comp) cudaStreamSynchronize(h->s_comp);
  if (h->s_h2d) cudaStreamSynchronize(h->s_h2d);
  if (h->s_d2h) cudaStreamSynchronize(h->s_d2h);
  for (int i = 0; i < 2; ++i) {
    if (h->ev_ready[i]) cudaEventDestroy(h->ev_ready[i]);
    if (h->ev_free[i]) cudaEventDestroy(h->ev_free[i]);
  }
  for (auto e : h->ev_slab_ready) if (e) cudaEventDestroy(e);
  for (auto e : h->ev_d2h_done) if (e) cudaEventDestroy(e);
  for (auto e : h->prof_events) if (e) cudaEventDestroy(e);
  if (h->prof_ref) cudaEventDestroy(h->prof_ref);
  for (int i = 0; i < 2; ++i)
    if (h->ev_loss[i]) cudaEventDestroy(h->ev_loss[i]);
  if (h->ev_resident) cudaEventDestroy(h->ev_resident);
  if (h->s_comp) cudaStreamDestroy(h->s_comp);
  if (h->s_h2d) cudaStreamDestroy(h->s_h2d);
  if (h->s_d2h) cudaStreamDestroy(h->s_d2h);
  if (h->dmem) cudaFree(h->dmem);
  if (h->store) cudaFreeHost(h->store);
  for (auto p : h->staging) if (p) cudaFreeHost(p);
  if (h->tok_pinned) cudaFreeHost(h->tok_pinned);
  if (h->loss_pinned) cudaFreeHost(h->loss_pinned);
  if (h->flag_pinned) cudaFreeHost(h->flag_pinned);
}

// Lay out all device buffers in one arena (first pass measures, second assigns).
void plan_device(mt_handle* h, Arena& A) {
  const size_t M = (size_t)h->Mmax, d = h->d, f = h->f, V = h->V, qn = h->qkvN, hq = h->hq;
  const size_t H = h->H;
  if (h->cfg.streamed) {
    h->wbuf[0] = take<bf16>(A, h->lay.max_unit);
    h->wbuf[1] = take<bf16>(A, h->lay.max_unit);
  } else {
    h->resident = take<bf16>(A, h->n_total);
  }
  h->slab.assign(h->cfg.n_slabs, nullptr);
  for (auto& p : h->slab) p = take<bf16>(A, h->lay.max_unit);
  h->d_tok = take<int32_t>(A, 2 * M);
  h->d_lab = h->d_tok + M;
  h->d_flag = take<int32_t>(A, 4);
  h->d_ework = take<int32_t>(A, (size_t)mt_k_embedding_bwd_work((int)M, (int)V));
  h->cos_t = take<float>(A, (size_t)h->cfg.max_seq * (h->hd / 2));
  h->sin_t = take<float>(A, (size_t)h->cfg.max_seq * (h->hd / 2));
  // xa holds the last layer's output; xb (with xa) the outputs inside a
  // segment of more than one layer
  h->xa = take<float>(A, M * d);
  h->xb = h->cfg.ckpt_interval > 1 ? take<float>(A, M * d) : nullptr;
  h->ckpt.assign(h->nseg, nullptr);
  for (auto& p : h->ckpt) p = take<float>(A, M * d);
  const int slots = std::min(h->cfg.ckpt_interval, h->L);
  h->saved.assign(slots, Saved{});
  for (int i = 0; i < slots; ++i) {
    Saved& S = h->saved[i];
    // the first layer of a segment reads its checkpoint in place
    S.x = i > 0 ? take<float>(A, M * d) : nullptr;
    S.u = take<bf16>(A, M * d);
    S.r1 = take<float>(A, M);
    S.qkv = take<bf16>(A, M * qn);
    // with keep_attention the layers' own kept tensors stand in for these
    S.o = h->cfg.keep_attention ? nullptr : take<bf16>(A, M * hq);
    S.lse = h->cfg.keep_attention ? nullptr : take<float>(A, M * H);
    S.h = take<float>(A, M * d);
    S.z = take<bf16>(A, M * d);
    S.r2 = take<float>(A, M);
    S.gu = take<bf16>(A, M * 2 * f);
    S.a = take<bf16>(A, M * f);
  }
  h->att_o.assign(h->cfg.keep_attention ? h->L : 0, nullptr);
  h->att_lse.assign(h->cfg.keep_attention ? h->L : 0, nullptr);
  for (int l = 0; l < (int)h->att_o.size(); ++l) {
    h->att_o[l] = take<bf16>(A, M * hq);
    h->att_lse[l] = take<float>(A, M * H);
  }
  h->xh = take<bf16>(A, M * d);
  h->rf = take<float>(A, M);
  h->logits = take<float>(A, (size_t)h->Mchunk * V);
  h->dz = take<bf16>(A, (h->dz_chunked ? (size_t)h->Mchunk : M) * V);
  h->dhead32 = h->dz_chunked ? take<float>(A, (size_t)V * d) : nullptr;
  h->loss_rows = take<float>(A, M);
  h->loss_dev = take<float>(A, 4);
  h->dx32 = take<float>(A, M * d);
  h->dh32 = take<float>(A, M * d);
  h->dn32 = take<float>(A, M * d);
  h->dxb = take<bf16>(A, M * d);
  h->dhb = take<bf16>(A, M * d);
  h->da = swiglu_bwd_fused(h) ? nullptr : take<bf16>(A, M * f);  // only the unfused SwiGLU backward
  h->dob = take<bf16>(A, M * hq);
  h->dqkv = take<bf16>(A, M * qn);
  h->delta = take<float>(A, M * H);
  {
    const int shp[5][2] = {{(int)d, (int)f}, {(int)(2 * f), (int)d}, {(int)d, (int)hq}, {(int)qn, (int)d}, {(int)V, (int)d}};
    size_t ws = 0;
    for (auto& x : shp) ws = std::max(ws, splitk_ws_elems(x[0], x[1]));
    h->wg_ws_elems = ws;
    h->wg_ws = ws ? take<float>(A, ws) : nullptr;
  }
  h->npart = take<float>(A, (size_t)mt_k_rmsnorm_bwd_parts((int)M) * d);

}

void set_dims(mt_handle* h, const mt_config& c) {
  h->L = c.n_layers;
  h->d = c.d_model;
  h->H = c.n_heads;
  h->Hkv = c.n_kv_heads;
  h->hd = c.head_dim;
  h->f = c.ffn_dim;
  h->V = c.vocab;
  h->qkvN = (h->H + 2 * h->Hkv) * h->hd;
  h->hq = h->H * h->hd;
  h->nseg = (h->L + c.ckpt_interval - 1) / c.ckpt_interval;
  h->Mmax = c.max_batch * c.max_seq;
  if (c.head_chunk_rows > 0) {
    h->Mchunk = (int)std::min<int64_t>(c.head_chunk_rows, h->Mmax);
    h->dz_chunked = h->Mchunk < h->Mmax;
  } else {
    int64_t mc = (1LL << 28) / h->V;
    mc = mc / 128 * 128;
    if (mc < 128) mc = 128;
    h->Mchunk = (int)std::min<int64_t>(mc, h->Mmax);
    // per-chunk dz only where it takes less memory than dz for every token
    const double full = 2.0 * h->Mmax * (double)h->V;
    const double chunked = 2.0 * h->Mchunk * (double)h->V + 4.0 * h->V * (double)h->d;
    h->dz_chunked = h->Mchunk < h->Mmax && chunked < full;
  }
}

int fail(mt_handle* h, int code, const std::string& msg) {
  set_err(h, msg);
  return code;
}

}  // namespace

void set_last_error_message(const std::string& msg) { g_thread_error = msg; }

}  // namespace mt

using namespace mt;

extern "C" {

int mt_layout(const mt_config* cfg, mt_tensor_desc* out, int cap, int* n_out, int64_t* n_total) {
  const char* why = nullptr;
  if (!cfg || !config_valid(*cfg, &why)) return fail(nullptr, MT_EINVAL, why ? why : "null config");
  FlatLayout L = build_layout(*cfg);
  const int n = (int)L.tensors.size();
  if (n_out) *n_out = n;
  if (n_total) *n_total = L.n_total;
  if (out) {
    for (int i = 0; i < n && i < cap; ++i) {
      const TensorDesc& t = L.tensors[i];
      out[i].unit = t.unit;
      out[i].kind = t.kind;
      out[i].offset = t.offset;
      out[i].rows = t.rows;
      out[i].cols = t.cols;
      std::memcpy(out[i].name, t.name, sizeof(out[i].name));
    }
  }
  return MT_OK;
}

int mt_unit_range(const mt_config* cfg, int unit, int64_t* offset, int64_t* length) {
  const char* why = nullptr;
  if (!cfg || !config_valid(*cfg, &why)) return fail(nullptr, MT_EINVAL, why ? why : "null config");
  if (unit < 0 || unit > cfg->n_layers + 1) return fail(nullptr, MT_EINVAL, "unit out of range");
  FlatLayout L = build_layout(*cfg);
  if (offset) *offset = L.unit_off[unit];
  if (length) *length = L.unit_len[unit];
  return MT_OK;
}

int mt_plan(const mt_config* cfg, int64_t* device_bytes, int64_t* pinned_bytes, int64_t* host_state_bytes) {
  const char* why = nullptr;
  if (!cfg || !config_valid(*cfg, &why)) return fail(nullptr, MT_EINVAL, why ? why : "null config");
  mt_handle h;
  h.cfg = *cfg;
  h.lay = build_layout(*cfg);
  h.n_total = h.lay.n_total;
  set_dims(&h, *cfg);
  try {
    Arena probe;
    probe.cap = ~size_t(0) >> 1;
    plan_device(&h, probe);
    if (device_bytes) *device_bytes = (int64_t)probe.used;
  } catch (const StepError& e) {
    return fail(nullptr, e.code, e.msg);
  }
  if (pinned_bytes)
    *pinned_bytes = (int64_t)(sizeof(uint16_t) * h.n_total + (size_t)cfg->n_slabs * sizeof(uint16_t) * h.lay.max_unit +
                              sizeof(int32_t) * 2 * (size_t)h.Mmax + sizeof(float) * 4 + sizeof(int32_t) * 4);
  if (host_state_bytes) *host_state_bytes = (int64_t)(4 * sizeof(float)) * h.n_total;
  return MT_OK;
}

int mt_debug_inject_global(int what, int64_t value) {
  if (what == 4) {
    g_fail_next_alloc.store(value ? 1 : 0);
    return MT_OK;
  }
  return MT_EINVAL;
}

int mt_init(const mt_config* cfg, float* master, float* adam_m, float* adam_v, float* grad, int64_t n_total,
            mt_handle** out) {
  if (!out) return fail(nullptr, MT_EINVAL, "null output handle");
  *out = nullptr;
  const char* why = nullptr;
  if (!cfg || !config_valid(*cfg, &why)) return fail(nullptr, MT_EINVAL, why ? why : "null config");
  if (!master || !adam_m || !adam_v) return fail(nullptr, MT_EINVAL, "null host state array");
  mt_handle* h = new (std::nothrow) mt_handle();
  if (!h) return fail(nullptr, MT_ENOMEM, "out of host memory");
  h->cfg = *cfg;
  h->lay = build_layout(*cfg);
  if (n_total != h->lay.n_total) {
    delete h;
    return fail(nullptr, MT_EINVAL, "n_total does not match the layout");
  }
  h->master = master;
  h->adam_m = adam_m;
  h->adam_v = adam_v;
  h->grad = grad;
  h->n_total = n_total;
  h->threads = cfg->host_threads > 0 ? cfg->host_threads : default_threads();
  set_dims(h, *cfg);
  try {
    if (g_fail_next_alloc.exchange(0)) throw StepError{MT_ENOMEM, "injected device allocation failure"};
    CK(cudaSetDevice(cfg->device));
    // device arena: measure, allocate, assign
    Arena probe;
    probe.cap = ~size_t(0) >> 1;
    plan_device(h, probe);
    Arena A;
    if (cudaMalloc(&h->dmem, probe.used) != cudaSuccess) {
      cudaGetLastError();
      throw StepError{MT_ENOMEM, "device allocation of " + std::to_string(probe.used) + " bytes failed"};
    }
    h->dbytes = probe.used;
    A.base = (uint8_t*)h->dmem;
    A.cap = probe.used;
    plan_device(h, A);
    // pinned host memory
    auto pin = [&](void** p, size_t bytes) {
      if (cudaHostAlloc(p, bytes, cudaHostAllocDefault) != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        throw StepError{MT_ENOMEM, "pinned allocation of " + std::to_string(bytes) + " bytes failed"};
      }
      h->st.pinned_bytes += (int64_t)bytes;
    };
    pin((void**)&h->store, sizeof(uint16_t) * n_total);
    h->staging.assign(cfg->n_slabs, nullptr);
    for (auto& p : h->staging) pin((void**)&p, sizeof(uint16_t) * h->lay.max_unit);
    pin((void**)&h->tok_pinned, sizeof(int32_t) * 2 * h->Mmax);
    pin((void**)&h->loss_pinned, sizeof(float) * 4);
    pin((void**)&h->flag_pinned, sizeof(int32_t) * 4);
    emit_bf16(master, h->store, n_total, h->threads);
    // streams and events
    CK(cudaStreamCreateWithFlags(&h->s_comp, cudaStreamNonBlocking));
    CK(cudaStreamCreateWithFlags(&h->s_h2d, cudaStreamNonBlocking));
    CK(cudaStreamCreateWithFlags(&h->s_d2h, cudaStreamNonBlocking));
    for (int i = 0; i < 2; ++i) {
      CK(cudaEventCreateWithFlags(&h->ev_ready[i], cudaEventDisableTiming));
      CK(cudaEventCreateWithFlags(&h->ev_free[i], cudaEventDisableTiming));
    }
    h->ev_slab_ready.assign(cfg->n_slabs, nullptr);
    h->ev_d2h_done.assign(cfg->n_slabs, nullptr);
    for (int k = 0; k < cfg->n_slabs; ++k) {
      CK(cudaEventCreateWithFlags(&h->ev_slab_ready[k], cudaEventDisableTiming));
      CK(cudaEventCreateWithFlags(&h->ev_d2h_done[k], cudaEventDisableTiming));
    }
    CK(cudaEventCreateWithFlags(&h->ev_loss[0], cudaEventDisableTiming));
    CK(cudaEventCreateWithFlags(&h->ev_loss[1], cudaEventDisableTiming));
    CK(cudaEventCreateWithFlags(&h->ev_resident, cudaEventDisableTiming));
    // RoPE tables in double precision on the host
    {
      const int half = h->hd / 2;
      std::vector<float> c((size_t)cfg->max_seq * half), s((size_t)cfg->max_seq * half);
      for (int t = 0; t < cfg->max_seq; ++t)
        for (int i = 0; i < half; ++i) {
          const double inv = std::pow((double)cfg->rope_theta, -2.0 * i / h->hd);
          const double ang = (double)t * inv;
          c[(size_t)t * half + i] = (float)std::cos(ang);
          s[(size_t)t * half + i] = (float)std::sin(ang);
        }
      CK(cudaMemcpy(h->cos_t, c.data(), sizeof(float) * c.size(), cudaMemcpyHostToDevice));
      CK(cudaMemcpy(h->sin_t, s.data(), sizeof(float) * s.size(), cudaMemcpyHostToDevice));
    }
    h->staging_busy.assign(cfg->n_slabs, 0);
    h->unit_pending.assign(h->L + 2, 0);
    h->st.device_bytes = (int64_t)h->dbytes;
    h->worker = std::thread(worker_main, h);
  } catch (const StepError& e) {
    set_err(nullptr, e.msg);
    destroy_resources(h);
    delete h;
    return e.code;
  } catch (const std::exception& e) {
    set_err(nullptr, e.what());
    destroy_resources(h);
    delete h;
    return MT_ENOMEM;
  }
  *out = h;
  return MT_OK;
}

static int run_step(mt_handle* h, const int32_t* tokens, const int32_t* labels, int B, int s, bool on_device,
                    float* loss_out, int micro_index = 0, int n_micro = 1) {
  if (!h) return fail(nullptr, MT_EINVAL, "null handle");
  if (h->broken) return fail(h, MT_ESTATE, "handle is unusable after an earlier timeout or device error");
  if (!tokens || !labels || B <= 0 || s <= 0 || B > h->cfg.max_batch || s > h->cfg.max_seq)
    return fail(h, MT_EINVAL, "bad tokens/labels or batch/seq outside the configured maxima");
  const int M = B * s;
  const auto t0 = Clock::now();
  if (n_micro < 1 || micro_index < 0 || micro_index >= n_micro)
    return fail(h, MT_EINVAL, "micro_index must lie in [0, n_micro)");
  if (n_micro > 1 && !h->grad)
    return fail(h, MT_ESTATE, "accumulation over micro-batches needs the FP32 gradient array at mt_init");
  Step st{h, B, s, M, h->t + 1};
  st.acc = micro_index > 0;
  st.adam = micro_index == n_micro - 1;
  st.gscale = 1.f / (float)n_micro;
  if (micro_index == 0) h->accum_nonfinite = false;
  try {
    CK(cudaSetDevice(h->cfg.device));
    if (!on_device) {
      for (int i = 0; i < M; ++i)
        if (tokens[i] < 0 || tokens[i] >= h->V || labels[i] < 0 || labels[i] >= h->V)
          return fail(h, MT_EINVAL, "token or label id outside [0, vocab)");
      std::memcpy(h->tok_pinned, tokens, sizeof(int32_t) * M);
      std::memcpy(h->tok_pinned + M, labels, sizeof(int32_t) * M);
      CK(cudaMemcpyAsync(h->d_tok, h->tok_pinned, sizeof(int32_t) * M, cudaMemcpyHostToDevice, h->s_comp));
      CK(cudaMemcpyAsync(h->d_lab, h->tok_pinned + M, sizeof(int32_t) * M, cudaMemcpyHostToDevice, h->s_comp));
    } else {
      CK(cudaMemcpyAsync(h->d_tok, tokens, sizeof(int32_t) * M, cudaMemcpyDeviceToDevice, h->s_comp));
      CK(cudaMemcpyAsync(h->d_lab, labels, sizeof(int32_t) * M, cudaMemcpyDeviceToDevice, h->s_comp));
      CK(cudaMemsetAsync(h->d_flag, 0, sizeof(int32_t), h->s_comp));
      KK(mt_k_check_ids(h->d_tok, 2 * M, h->V, h->d_flag, h->s_comp));
      CK(cudaMemcpyAsync(h->flag_pinned, h->d_flag, sizeof(int32_t), cudaMemcpyDeviceToHost, h->s_comp));
      CK(cudaStreamSynchronize(h->s_comp));
      if (*h->flag_pinned) return fail(h, MT_EDEVICE, "token or label id outside [0, vocab) (device check)");
    }
    {
      std::lock_guard<std::mutex> lk(h->mu);
      if (h->worker_error) {
        // an overlapped Adam of the previous step failed: report it now
        const int code = h->worker_error;
        h->worker_error = 0;
        return fail(h, code, h->worker_msg);
      }
      h->units_done = 0;
      h->worker_msg.clear();
    }
    st.run();
    if (!h->cfg.overlap_adam) {
      // wait for the worker to finish every unit of this step
      std::unique_lock<std::mutex> lk(h->mu);
      const bool ok = h->cv.wait_for(lk, std::chrono::milliseconds(h->deadline_ms),
                                     [&] { return h->units_done == h->L + 2 || h->worker_error; });
      if (h->worker_error) throw StepError{h->worker_error, h->worker_msg};
      if (!ok) throw StepError{MT_ETIMEOUT, "timed out waiting for the host optimizer"};
    }
    CK(cudaStreamSynchronize(h->s_comp));
    CK(cudaStreamSynchronize(h->s_d2h));
    CK(cudaStreamSynchronize(h->s_h2d));
    if (h->prof_on) {
      h->timeline.clear();
      h->timeline_seq = h->step_seq;
      for (size_t i = 0; i < h->prof_recs.size(); ++i) {
        float ms = 0.f, t0 = 0.f, t1 = 0.f;
        CK(cudaEventElapsedTime(&ms, h->prof_events[2 * i], h->prof_events[2 * i + 1]));
        const auto& r = h->prof_recs[i];
        h->prof.ms[r.cat] += ms;
        h->prof.flops[r.cat] += r.flops;
        h->prof.bytes[r.cat] += r.bytes;
        if (h->prof_ref) {
          CK(cudaEventElapsedTime(&t0, h->prof_ref, h->prof_events[2 * i]));
          CK(cudaEventElapsedTime(&t1, h->prof_ref, h->prof_events[2 * i + 1]));
          h->timeline.push_back(mt_timeline_rec{r.cat, r.stream, (double)t0, (double)t1});
        }
      }
    }
    h->prof_recs.clear();
    int dev_err = 0;
    if (mt_k_device_error(&dev_err, 1) != MT_OK) throw StepError{MT_ECUDA, "reading the device error word failed"};
    if (dev_err) throw StepError{MT_EDEVICE, "a kernel reported device error " + std::to_string(dev_err)};
  } catch (const StepError& e) {
    // drain: nothing may stay in flight when the call returns
    cudaStreamSynchronize(h->s_comp);
    cudaStreamSynchronize(h->s_h2d);
    cudaStreamSynchronize(h->s_d2h);
    std::unique_lock<std::mutex> lk(h->mu);
    h->jobs.clear();
    const bool idle = h->cv.wait_for(lk, std::chrono::milliseconds(std::min<int64_t>(h->deadline_ms, 60000)),
                                     [&] { return h->in_flight == 0; });
    if (e.code == MT_ETIMEOUT || e.code == MT_EDEVICE || e.code == MT_ECUDA || !idle) h->broken = 1;
    if (idle) std::fill(h->unit_pending.begin(), h->unit_pending.end(), 0);
    h->worker_error = 0;  // reported by this call
    for (auto& b : h->staging_busy) b = 0;
    h->prof_recs.clear();
    h->err = e.msg;
    g_thread_error = e.msg;
    return e.code;
  }
  const float total = h->loss_pinned[st.parity()];
  const float loss = total / (float)M;
  if (loss_out) *loss_out = loss;
  h->st.steps += 1;
  h->st.last_step_s = seconds_since(t0);
  if (!std::isfinite(total)) {
    h->accum_nonfinite = true;
    return fail(h, MT_ENONFINITE, "non-finite loss: no Adam update was applied");
  }
  if (st.adam && !h->accum_nonfinite) h->t += 1;
  return MT_OK;
}

int mt_train_step(mt_handle* h, const int32_t* tokens, const int32_t* labels, int32_t batch, int32_t seq,
                  float* loss_out) {
  return run_step(h, tokens, labels, batch, seq, false, loss_out);
}

int mt_train_step_device(mt_handle* h, const int32_t* d_tokens, const int32_t* d_labels, int32_t batch, int32_t seq,
                         float* loss_out) {
  return run_step(h, d_tokens, d_labels, batch, seq, true, loss_out);
}

int mt_train_step_accum(mt_handle* h, const int32_t* tokens, const int32_t* labels, int32_t batch, int32_t seq,
                        int32_t micro_index, int32_t n_micro, float* loss_out) {
  return run_step(h, tokens, labels, batch, seq, false, loss_out, micro_index, n_micro);
}

int mt_sync(mt_handle* h) {
  if (!h) return fail(nullptr, MT_EINVAL, "null handle");
  std::unique_lock<std::mutex> lk(h->mu);
  const bool ok = h->cv.wait_for(lk, std::chrono::milliseconds(h->deadline_ms),
                                 [&] { return (h->jobs.empty() && h->in_flight == 0) || h->worker_error; });
  if (h->worker_error) {
    const int code = h->worker_error;
    h->worker_error = 0;
    h->err = h->worker_msg;
    g_thread_error = h->worker_msg;
    return code;
  }
  if (!ok) {
    h->err = "timed out waiting for the host optimizer";
    g_thread_error = h->err;
    return MT_ETIMEOUT;
  }
  return MT_OK;
}

int mt_read_grads(mt_handle* h, float* dst, int64_t n) {
  if (!h || !dst || n < 0 || n > h->n_total) return fail(h, MT_EINVAL, "bad arguments to mt_read_grads");
  if (!h->grad) return fail(h, MT_ESTATE, "no FP32 gradient array: gradients went straight into Adam");
  if (const int r = mt_sync(h)) return r;
  if (dst != h->grad) std::memcpy(dst, h->grad, sizeof(float) * n);
  return MT_OK;
}

int mt_get_step(mt_handle* h, int64_t* t) {
  if (!h || !t) return MT_EINVAL;
  *t = h->t;
  return MT_OK;
}

int mt_set_step(mt_handle* h, int64_t t) {
  if (!h || t < 0) return MT_EINVAL;
  if (const int r = mt_sync(h)) return r;
  h->t = t;
  return MT_OK;
}

int mt_sync_store(mt_handle* h) {
  if (!h) return MT_EINVAL;
  if (const int r = mt_sync(h)) return r;
  emit_bf16(h->master, h->store, h->n_total, h->threads);
  return MT_OK;
}

int mt_get_stats(mt_handle* h, mt_stats* out) {
  if (!h || !out) return MT_EINVAL;
  std::lock_guard<std::mutex> lk(h->mu);
  *out = h->st;
  return MT_OK;
}

int mt_get_stream(mt_handle* h, int which, void** stream) {
  if (!h || !stream || which < 0 || which > 2) return MT_EINVAL;
  *stream = which == 0 ? (void*)h->s_comp : which == 1 ? (void*)h->s_h2d : (void*)h->s_d2h;
  return MT_OK;
}

int mt_profile_enable(mt_handle* h, int on) {
  if (!h) return MT_EINVAL;
  h->prof_on = on ? 1 : 0;
  return MT_OK;
}

int mt_profile_read(mt_handle* h, mt_kernel_profile* out, int reset) {
  if (!h || !out) return MT_EINVAL;
  *out = h->prof;
  if (reset) h->prof = mt_kernel_profile{};
  return MT_OK;
}

int mt_profile_timeline(mt_handle* h, mt_timeline_rec* out, int cap, int* n_out) {
  if (!h || !n_out || cap < 0 || (cap > 0 && !out)) return MT_EINVAL;
  std::vector<mt_timeline_rec> all = h->timeline;
  {
    std::lock_guard<std::mutex> lk(h->mu);
    if (h->host_tl_seq == h->timeline_seq) {
      all.insert(all.end(), h->host_tl.begin(), h->host_tl.end());
      // the previous step's worker intervals that run into this step (its
      // host tail under overlap_adam), on this step's clock, as streams 5, 6
      if (h->host_tl_prev_seq == h->timeline_seq - 1) {
        const double dt =
            std::chrono::duration<double, std::milli>(h->host_tl_prev_step0 - h->host_tl_step0).count();
        for (const auto& r : h->host_tl_prev)
          if (r.end_ms + dt > 0.0) all.push_back(mt_timeline_rec{r.cls, r.stream + 2, r.start_ms + dt, r.end_ms + dt});
      }
    }
  }
  const int n = (int)all.size();
  for (int i = 0; i < n && i < cap; ++i) out[i] = all[i];
  *n_out = n;
  return MT_OK;
}

int mt_destroy(mt_handle* h) {
  if (!h) return MT_EINVAL;
  destroy_resources(h);
  delete h;
  return MT_OK;
}

const char* mt_last_error(mt_handle* h) { return h ? h->err.c_str() : g_thread_error.c_str(); }

int mt_debug_inject(mt_handle* h, int what, int64_t value) {
  if (!h) return MT_EINVAL;
  std::lock_guard<std::mutex> lk(h->mu);
  switch (what) {
    case 1: h->inject_sleep_ms = value; return MT_OK;
    case 2: h->inject_fail_at = value > 0 ? h->worker_units_total + value : 0; return MT_OK;
    case 3: h->deadline_ms = value > 0 ? value : 600000; return MT_OK;
    default: return MT_EINVAL;
  }
}

int mt_host_adam(float* w, float* m, float* v, const float* g, uint16_t* store, int64_t n, int64_t t, float lr,
                 float beta1, float beta2, float eps, int threads) {
  if (!w || !m || !v || !g || n < 0 || t < 1) return MT_EINVAL;
  AdamArgs a{};
  a.w = w;
  a.m = m;
  a.v = v;
  a.grad_out = nullptr;
  a.grad_in = g;
  a.slab = nullptr;
  a.store = store;
  a.n = n;
  a.t = t;
  a.lr = lr;
  a.beta1 = beta1;
  a.beta2 = beta2;
  a.eps = eps;
  a.apply = true;
  adam_pass(a, threads > 0 ? threads : default_threads());
  return MT_OK;
}

int mt_host_adam_slab(float* w, float* m, float* v, const uint16_t* slab, float* grad_out, uint16_t* store,
                      int64_t n, int64_t t, float lr, float beta1, float beta2, float eps, int threads) {
  if (!w || !m || !v || !slab || n < 0 || t < 1) return MT_EINVAL;
  AdamArgs a{};
  a.w = w;
  a.m = m;
  a.v = v;
  a.grad_out = grad_out;
  a.grad_in = nullptr;
  a.slab = slab;
  a.store = store;
  a.n = n;
  a.t = t;
  a.lr = lr;
  a.beta1 = beta1;
  a.beta2 = beta2;
  a.eps = eps;
  a.apply = true;
  adam_pass(a, threads > 0 ? threads : default_threads());
  return MT_OK;
}

int mt_host_to_bf16(const float* src, uint16_t* dst, int64_t n) {
  if (!src || !dst || n < 0) return MT_EINVAL;
  emit_bf16(src, dst, n, default_threads());
  return MT_OK;
}

}  // extern "C"
