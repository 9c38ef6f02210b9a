/*
 * mt.h - C ABI of the streamed-layer training step (libmt.so).
 *
 * One training step of a Llama-style decoder whose persistent state lives in
 * host memory, as the RAM-centric training articles describe:
 *
 *  - "MegaTrain：单卡训百亿大模型的突破与实践" (zhichai.net), section
 *    "以内存为中心的训练新范式": parameters, gradients and Adam moments stay
 *    in host RAM (point 1); layers are prefetched into two ping-pong device
 *    buffers and released after use, gradients go back layer by layer
 *    (point 2); activations are checkpointed every few layers and recomputed
 *    (point 3); a stateless layer template runs each layer (point 4).
 *  - lqnn.cn MegaTrain article, section 三: "gpu_flat_buffers" (two fixed
 *    device flat buffers), "layer_pinned_flats" (pinned flat per-layer
 *    weights), three CUDA streams gated by weight_ready / buffer_free events,
 *    a K-slab flat gradient pool drained by a CPU worker thread that adds the
 *    slabs into FP32 master gradients, checkpoint_interval (default 4);
 *    section 二: ParameterState = FP32 master, grad, m, v; Adam runs on the CPU.
 *
 * Every function returns MT_OK (0) or a negative MT_E* code; no C++
 * exception crosses this boundary and nothing aborts. After any error the
 * handle can still be destroyed. mt_last_error() gives a text message.
 */
#ifndef MT_H_
#define MT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MT_OK 0
#define MT_EINVAL (-1)     /* bad argument, shape or token id; nothing ran */
#define MT_ENOMEM (-2)     /* host or device allocation failed */
#define MT_ECUDA (-3)      /* a CUDA runtime call failed */
#define MT_ETIMEOUT (-4)   /* a host wait (worker, event) passed its deadline */
#define MT_EWORKER (-5)    /* the host worker thread failed */
#define MT_ENONFINITE (-6) /* the loss was NaN or Inf; master/m/v were not updated */
#define MT_ESTATE (-7)     /* handle in a state that forbids the call */
#define MT_EDEVICE (-8)    /* a kernel recorded an error in the device error word */

/* Model shape and run settings. All counts are positive. */
typedef struct mt_config {
  int32_t n_layers;      /* L */
  int32_t d_model;       /* d, multiple of 64 */
  int32_t n_heads;       /* H */
  int32_t n_kv_heads;    /* Hkv, divides H */
  int32_t head_dim;      /* hd in {16, 64, 128} */
  int32_t ffn_dim;       /* f, multiple of 64 */
  int32_t vocab;         /* V, multiple of 8 */
  int32_t max_batch;     /* largest B a step may use */
  int32_t max_seq;       /* largest s a step may use */
  int32_t ckpt_interval; /* C >= 1: checkpoint the input of every C-th layer */
  int32_t n_slabs;       /* K >= 2 gradient slabs (device + pinned host staging) */
  int32_t streamed;      /* 1: stream units through two buffers; 0: all units resident */
  float rms_eps;         /* RMSNorm epsilon, e.g. 1e-5 */
  float rope_theta;      /* RoPE base, e.g. 10000 */
  float lr, beta1, beta2, adam_eps; /* Adam, no weight decay */
  int32_t device;        /* CUDA device ordinal */
  int32_t host_threads;  /* threads for host accumulate + Adam; 0 = every core */
  int32_t overlap_adam;  /* 1: mt_train_step returns once the device work and the loss are done while
                            the host worker finishes Adam on the last units; the next step uploads each
                            unit only after its Adam has finished. Results are identical to 0. Call
                            mt_sync before reading master / m / v yourself. */
  int32_t unfused_epilogues; /* 1: RoPE and SwiGLU (forward and backward) run as separate kernels
                                after their GEMMs, which round the GEMM output to bf16 first; 0 (the
                                default, faster): the GEMM epilogues apply them to the fp32 product and
                                round once. Both match the same bars against the exact step */
  int32_t keep_attention;    /* 1: keep every layer's attention output and log-sum-exp from the
                                forward (L * (M * H * hd * 2 + M * H * 4) more device bytes) so the
                                backward's recompute skips the attention core; results are bitwise
                                identical. 0 (default): recompute whole layers from the checkpoints */
  int32_t head_chunk_rows;   /* rows of one logits chunk of the head. 0 (default): about 2^28 / V
                                rows, and the head's gradient dz is kept per chunk (the head's weight
                                gradient summed over chunks in fp32) only where that takes less
                                memory than dz for every token; > 0: chunks of this many rows, dz
                                per chunk whenever there is more than one chunk */
} mt_config;

/* One tensor of the flat layout. kind 0 = matrix, 1 = norm weight. */
typedef struct mt_tensor_desc {
  int32_t unit;   /* 0 = embedding, 1..L = layer l-1, L+1 = final norm + head */
  int32_t kind;
  int64_t offset; /* absolute element offset in the flat arrays */
  int64_t rows, cols; /* matrices [out, in]; vectors have cols = 1 */
  char name[24];
} mt_tensor_desc;

typedef struct mt_stats {
  int64_t steps;
  int64_t h2d_bytes;       /* weight bytes copied host->device, all steps */
  int64_t d2h_bytes;       /* gradient bytes copied device->host, all steps */
  int64_t h2d_units;       /* unit copies issued (forward + recompute) */
  double host_adam_s;      /* worker time in accumulate + Adam + bf16 emit */
  double host_wait_s;      /* main-thread time blocked on slab back-pressure */
  double last_step_s;      /* wall time of the last mt_train_step */
  int64_t device_bytes;    /* device memory owned by the handle */
  int64_t pinned_bytes;    /* pinned host memory owned by the handle */
  int64_t kernel_launches; /* kernels launched by the handle, all steps */
  double host_compute_s;   /* worker time inside accumulate + Adam + emit only */
  double host_copy_wait_s; /* worker time waiting for slab copies and the loss */
} mt_stats;

/* Kernel classes of the per-kernel profile. */
#define MT_PROF_GEMM 0
#define MT_PROF_ATTN_FWD 1
#define MT_PROF_ATTN_BWD 2
#define MT_PROF_NORM 3
#define MT_PROF_ROPE 4
#define MT_PROF_SWIGLU 5
#define MT_PROF_RESERVED 6  /* no kernel of the step falls in this class */
#define MT_PROF_CE 7
#define MT_PROF_EMBED 8
#define MT_PROF_OTHER 9
#define MT_PROF_H2D 10   /* weight-unit copies, host store -> device buffer */
#define MT_PROF_D2H 11   /* gradient-slab copies, device slab -> pinned staging */
#define MT_PROF_N 12

/* Per-class totals: launches, device time (CUDA events around each launch
 * on the compute stream, only while profiling is enabled), algorithmic
 * FLOPs and algorithmic HBM bytes of the timed launches. The two copy
 * classes count copies instead of launches, time them with events on their
 * own streams, and give the bytes copied. */
typedef struct mt_kernel_profile {
  int64_t launches[MT_PROF_N];
  double ms[MT_PROF_N];
  double flops[MT_PROF_N];
  double bytes[MT_PROF_N];
} mt_kernel_profile;

typedef struct mt_handle mt_handle;

/*
 * Flat layout of `cfg` (no GPU needed). Writes up to `cap` descriptors and
 * the total element count n_total (tensor offsets are multiples of 64; the
 * padding counts). Order: embed; per layer attn_norm, wqkv, wo, mlp_norm,
 * wgu, wdown; final_norm, head. Returns MT_EINVAL on a bad shape.
 */
int mt_layout(const mt_config* cfg, mt_tensor_desc* out, int cap, int* n_out, int64_t* n_total);

/* Element range [offset, offset + length) of unit `unit` (0 .. L+1). */
int mt_unit_range(const mt_config* cfg, int unit, int64_t* offset, int64_t* length);

/*
 * Memory plan of `cfg` without a GPU and without allocating: device bytes of
 * the handle's arena (weight buffers, slabs, checkpoints, activations,
 * scratch; the same planner mt_init uses), pinned host bytes (bf16 store,
 * staging slabs, token staging) and the caller's FP32 state with the
 * gradient array (master, m, v, grad = 16 bytes per element; 12 without
 * the gradient array). Any pointer may be NULL.
 */
int mt_plan(const mt_config* cfg, int64_t* device_bytes, int64_t* pinned_bytes, int64_t* host_state_bytes);

/*
 * Creates a handle. master, adam_m, adam_v, grad are caller-owned FP32 host
 * arrays of n_total elements in the flat layout; they must stay valid until
 * mt_destroy. The caller initialises master and zeroes m and v. grad may be
 * NULL: each unit's bf16 gradient then goes straight from its staging slab
 * into Adam (the same arithmetic; the host holds FP32 master, m and v, the
 * 12 bytes per parameter of the lqnn.cn article's section 一, and no FP32
 * gradient stream crosses host memory); mt_read_grads then returns
 * MT_ESTATE and mt_train_step_accum accepts only n_micro = 1. The library
 * allocates the pinned bf16 flat store (filled with round-to-nearest-even
 * bf16 of master), the pinned staging slabs, all device memory and the
 * three streams, and starts the host worker thread. Returns MT_ENOMEM,
 * MT_ECUDA or MT_EINVAL on failure (nothing leaks).
 */
int mt_init(const mt_config* cfg, float* master, float* adam_m, float* adam_v, float* grad, int64_t n_total,
            mt_handle** out);

/*
 * One training step on host token and label arrays (int32 [batch, seq],
 * row-major, every id in [0, V), read only during the call). Computes the
 * mean cross-entropy loss of the current master (written to *loss_out),
 * overwrites `grad` with this step's FP32 gradient, and applies one Adam step
 * (t += 1) to master / m / v and to the bf16 store. Returns after all of it
 * is done. On MT_ENONFINITE the gradient is written but no Adam update
 * happens.
 */
int mt_train_step(mt_handle* h, const int32_t* tokens, const int32_t* labels, int32_t batch, int32_t seq,
                  float* loss_out);

/* Same as mt_train_step with tokens and labels already in device memory
 * (int32 [batch, seq]); ids are checked on the device and a bad id returns
 * MT_EDEVICE before any weight is touched by Adam. */
int mt_train_step_device(mt_handle* h, const int32_t* d_tokens, const int32_t* d_labels, int32_t batch,
                         int32_t seq, float* loss_out);

/*
 * Gradient accumulation over micro-batches (a way the travelaiplan blog,
 * "怎麼開始" step 3, suggests to grow the global batch): micro_index runs
 * 0 .. n_micro-1. Micro-step 0 sets the FP32 gradient to its micro-batch
 * gradient, later ones add theirs; the last one divides the sum by n_micro
 * (so `grad` holds the mean, the gradient of the mean loss over all
 * micro-batches of equal size) and applies one Adam step (t += 1). A
 * non-finite loss in any micro-step skips that Adam step. mt_train_step is
 * the n_micro = 1 case. n_micro > 1 needs the gradient array (MT_ESTATE
 * without it).
 */
int mt_train_step_accum(mt_handle* h, const int32_t* tokens, const int32_t* labels, int32_t batch, int32_t seq,
                        int32_t micro_index, int32_t n_micro, float* loss_out);

/* Copies the FP32 gradient of the last step (n elements, n <= n_total).
 * MT_ESTATE when the handle was created without a gradient array. */
int mt_read_grads(mt_handle* h, float* dst, int64_t n);

/* Waits until the host worker has finished every queued unit (Adam of the
 * last step included); returns a worker error if one occurred. Needed only
 * with overlap_adam = 1, before reading master / m / v / grad directly. */
int mt_sync(mt_handle* h);

int mt_get_step(mt_handle* h, int64_t* t);
int mt_set_step(mt_handle* h, int64_t t);     /* for resume from a checkpoint */
/* Re-emits the bf16 store from master (after the caller rewrote master). */
int mt_sync_store(mt_handle* h);
int mt_get_stats(mt_handle* h, mt_stats* out);
/* Returns the handle's CUDA stream: which 0 = compute, 1 = H2D, 2 = D2H. */
int mt_get_stream(mt_handle* h, int which, void** stream);
/* Brackets every kernel launch of later steps with CUDA events on the
 * compute stream (on = 1) so mt_profile_read() can report device time per
 * kernel class; adds two event records per launch. */
int mt_profile_enable(mt_handle* h, int on);
/* Copies the accumulated per-class profile; reset = 1 clears it. */
int mt_profile_read(mt_handle* h, mt_kernel_profile* out, int reset);

/* One interval of the last profiled step, in ms after the step began (a
 * copy may start before: negative). stream 0, 1, 2: a launch on the compute
 * stream or a copy on the host-to-device or device-to-host stream, timed
 * with CUDA events from the step's first compute-stream event; cls is its
 * MT_PROF_* class. stream 3: the host worker's accumulate + Adam pass over
 * unit cls; stream 4: the worker waiting for that unit's slab copy (host
 * clock from the start of the mt_train_step call); streams 5, 6: the same
 * for units of the step before that ran into this one (its host tail when
 * overlap_adam = 1), on this step's clock. */
typedef struct mt_timeline_rec {
  int32_t cls;
  int32_t stream;
  double start_ms, end_ms;
} mt_timeline_rec;

/* Copies up to `cap` records of the last step run with profiling enabled
 * (in issue order) into `out` and sets *n_out to their total number (call
 * with cap = 0 to size the buffer). No records before a profiled step. */
int mt_profile_timeline(mt_handle* h, mt_timeline_rec* out, int cap, int* n_out);
int mt_destroy(mt_handle* h);
/* Last error message of `h`, or of the calling thread when h is NULL. */
const char* mt_last_error(mt_handle* h);

/*
 * Host-side fault injection for tests (no GPU fault is ever caused):
 *  what 1: the worker sleeps `value` ms before each unit (deadline tests);
 *  what 2: the worker reports a failure on its `value`-th unit;
 *  what 3: host wait deadline in ms (default 600000);
 *  what 4: next device allocation in mt_init fails (value 1).
 */
int mt_debug_inject(mt_handle* h, int what, int64_t value);
/* Global (pre-handle) injection: what 4 = fail the next mt_init allocation. */
int mt_debug_inject_global(int what, int64_t value);

/*
 * Host Adam of the library on caller arrays (n elements, step t >= 1), the
 * same code the worker runs per unit: m, v, w updated in place; `g` FP32;
 * `store` (may be NULL) receives bf16(w) with round-to-nearest-even.
 */
int mt_host_adam(float* w, float* m, float* v, const float* g, uint16_t* store, int64_t n, int64_t t, float lr,
                 float beta1, float beta2, float eps, int threads);

/*
 * The worker's per-unit pass on caller arrays: gradient from a bf16 slab
 * (`slab`, n elements), written as FP32 to `grad_out` (may be NULL), then
 * Adam on w / m / v and the bf16 emit into `store` (may be NULL). The
 * slab accumulation of the lqnn.cn article's section 三.3 fused with the
 * host Adam of its section 二.
 */
int mt_host_adam_slab(float* w, float* m, float* v, const uint16_t* slab, float* grad_out, uint16_t* store,
                      int64_t n, int64_t t, float lr, float beta1, float beta2, float eps, int threads);

/* Round-to-nearest-even FP32 -> bf16 bits on the host; every NaN becomes 0x7fc0. */
int mt_host_to_bf16(const float* src, uint16_t* dst, int64_t n);

#ifdef __cplusplus
}
#endif
#endif /* MT_H_ */
