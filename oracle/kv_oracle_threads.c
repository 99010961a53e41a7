/*
 * Host-thread runner for the CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * Times the oracle's write loops (kv_oracle.c, unchanged) on several POSIX
 * threads for the benchmark's CPU-baseline leg and reference arm.  Tokens are
 * independent in both pages' write paths (sglang kvcache.cuh `store_kvcache`
 * and trtllm_fp8_kv_kernel.py `_fused_fp8_set_kv_buffer_kernel` handle each
 * token on its own), so thread i takes the token range
 * [T*i/n, T*(i+1)/n) and calls the oracle function on it.  Running the split
 * here rather than from Python keeps the interpreter lock out of the timed
 * loop.  Nothing in this file computes any part of the write path.
 */
#define _POSIX_C_SOURCE 200809L
#include <pthread.h>
#include <stdint.h>
#include <time.h>

int kvo_store_copy(const uint8_t *k, const uint8_t *v, uint8_t *k_cache, uint8_t *v_cache,
                   const void *indices, int index_is_i64, int64_t index_stride,
                   int64_t t_begin, int64_t t_end, int32_t num_heads, int32_t head_dim,
                   int32_t elem_bytes, const int64_t *strides, int64_t size_limit,
                   int64_t *bad_count, int64_t *first_bad);
int kvo_store_copy_paged(const uint8_t *k, const uint8_t *v, uint8_t *k_cache, uint8_t *v_cache,
                         const void *indices, int index_is_i64, int64_t index_stride,
                         int64_t t_begin, int64_t t_end, int32_t num_heads, int32_t head_dim,
                         int32_t elem_bytes, const int64_t *strides, int64_t page_size,
                         int64_t kc_page_stride, int64_t vc_page_stride, int64_t size_limit,
                         int64_t *bad_count, int64_t *first_bad);
int kvo_store_fp8(const uint8_t *k, const uint8_t *v, uint8_t *k_cache, uint8_t *v_cache,
                  const void *indices, int index_is_i64, int64_t index_stride,
                  int64_t t_begin, int64_t t_end, int32_t num_heads, int32_t head_dim,
                  int src_is_bf16, const int64_t *strides, int64_t page_size,
                  int64_t kc_page_stride, int64_t vc_page_stride, int64_t size_limit,
                  float inv_k, float inv_v, int use_scale,
                  int64_t *bad_count, int64_t *first_bad);

#define KVO_JOB_COPY 0
#define KVO_JOB_COPY_PAGED 1
#define KVO_JOB_FP8 2
#define KVO_MAX_THREADS 1024

/* One write problem: the arguments of the oracle call it names.  `dtype` is
 * elem_bytes for the copies and src_is_bf16 for the FP8 write. */
typedef struct kvo_job {
    int32_t kind;
    int32_t index_is_i64;
    const uint8_t *k, *v;
    uint8_t *k_cache, *v_cache;
    const void *indices;
    int64_t index_stride;
    int32_t num_heads, head_dim, dtype, use_scale;
    const int64_t *strides;
    int64_t page_size, kc_page_stride, vc_page_stride, size_limit;
    float inv_k, inv_v;
} kvo_job;

typedef struct worker {
    const kvo_job *job;
    int64_t t0, t1, min_reps, reps, bad;
    double seconds, end;
    const double *start;
    struct gate *gate;
    int rc;
} worker;

/* Start line: the workers wait until the runner opens it. */
struct gate {
    pthread_mutex_t m;
    pthread_cond_t c;
    int open;
};

static double now_s(void)
{
    struct timespec ts;
    clock_gettime(CLOCK_MONOTONIC, &ts);
    return (double)ts.tv_sec + 1e-9 * (double)ts.tv_nsec;
}

static int run_range(const kvo_job *j, int64_t t0, int64_t t1, int64_t *bad)
{
    int64_t first = -1;
    switch (j->kind) {
    case KVO_JOB_COPY:
        return kvo_store_copy(j->k, j->v, j->k_cache, j->v_cache, j->indices, j->index_is_i64,
                              j->index_stride, t0, t1, j->num_heads, j->head_dim, j->dtype,
                              j->strides, j->size_limit, bad, &first);
    case KVO_JOB_COPY_PAGED:
        return kvo_store_copy_paged(j->k, j->v, j->k_cache, j->v_cache, j->indices,
                                    j->index_is_i64, j->index_stride, t0, t1, j->num_heads,
                                    j->head_dim, j->dtype, j->strides, j->page_size,
                                    j->kc_page_stride, j->vc_page_stride, j->size_limit, bad,
                                    &first);
    case KVO_JOB_FP8:
        return kvo_store_fp8(j->k, j->v, j->k_cache, j->v_cache, j->indices, j->index_is_i64,
                             j->index_stride, t0, t1, j->num_heads, j->head_dim, j->dtype,
                             j->strides, j->page_size, j->kc_page_stride, j->vc_page_stride,
                             j->size_limit, j->inv_k, j->inv_v, j->use_scale, bad, &first);
    default:
        return 1;
    }
}

static void *work(void *arg)
{
    worker *w = (worker *)arg;
    pthread_mutex_lock(&w->gate->m);
    while (!w->gate->open)
        pthread_cond_wait(&w->gate->c, &w->gate->m);
    pthread_mutex_unlock(&w->gate->m);
    const double deadline = *w->start + w->seconds;
    for (;;) {
        int64_t bad = 0;
        w->rc |= run_range(w->job, w->t0, w->t1, &bad);
        w->bad += bad;
        w->reps += 1;
        const double t = now_s();
        if (w->rc != 0 || (t >= deadline && w->reps >= w->min_reps)) {
            w->end = t;
            return NULL;
        }
    }
}

/* Runs `job` over tokens [0, num_tokens) on `nthreads` threads, each thread
 * repeating its own token range until `seconds` have passed and it has done
 * at least `min_reps` passes (seconds = 0, min_reps = 1: one pass over the
 * batch).  *tokens_done = tokens processed by all threads; *elapsed = seconds
 * from the common start to the last thread's end; *bad_tokens = out-of-range
 * slots met.  Returns 0, or 1 for bad arguments or an oracle error. */
int kvo_run_threads(const kvo_job *job, int64_t num_tokens, int32_t nthreads, double seconds,
                    int64_t min_reps, int64_t *tokens_done, double *elapsed, int64_t *bad_tokens)
{
    if (!job || num_tokens < 1 || nthreads < 1 || min_reps < 1 || seconds < 0)
        return 1;
    if (nthreads > num_tokens)
        nthreads = (int32_t)num_tokens;
    if (nthreads > KVO_MAX_THREADS)
        nthreads = KVO_MAX_THREADS;
    static pthread_mutex_t lock = PTHREAD_MUTEX_INITIALIZER;
    pthread_mutex_lock(&lock);   /* one run at a time: the workers live on this stack */
    worker ws[KVO_MAX_THREADS];
    pthread_t th[KVO_MAX_THREADS];
    struct gate gate = {PTHREAD_MUTEX_INITIALIZER, PTHREAD_COND_INITIALIZER, 0};
    double start = 0.0;
    int started = 0, rc = 0;
    for (int i = 0; i < nthreads; ++i) {
        worker *w = &ws[i];
        w->job = job;
        w->t0 = num_tokens * i / nthreads;
        w->t1 = num_tokens * (i + 1) / nthreads;
        w->min_reps = min_reps;
        w->reps = 0;
        w->bad = 0;
        w->seconds = seconds;
        w->end = 0.0;
        w->start = &start;
        w->gate = &gate;
        w->rc = 0;
        if (pthread_create(&th[i], NULL, work, w) != 0) {
            rc = 1;   /* the threads that did start still run; the call reports the failure */
            break;
        }
        ++started;
    }
    pthread_mutex_lock(&gate.m);
    start = now_s();
    gate.open = 1;
    pthread_cond_broadcast(&gate.c);
    pthread_mutex_unlock(&gate.m);
    int64_t tokens = 0, bad = 0;
    double last = start;
    for (int i = 0; i < started; ++i) {
        pthread_join(th[i], NULL);
        rc |= ws[i].rc;
        tokens += ws[i].reps * (ws[i].t1 - ws[i].t0);
        bad += ws[i].bad;
        if (ws[i].end > last) last = ws[i].end;
    }
    pthread_mutex_unlock(&lock);
    if (tokens_done) *tokens_done = tokens;
    if (elapsed) *elapsed = last - start;
    if (bad_tokens) *bad_tokens = bad;
    return rc;
}
