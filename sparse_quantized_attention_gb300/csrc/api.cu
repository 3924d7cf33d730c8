// api.cu -- the C ABI of libffd.so (declared in include/ffd.h): argument checks, workspace
// planning and kernel launches. No function here allocates device memory.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

#include <cudaTypedefs.h>

namespace ffd {
cudaError_t launch_quantize(int P, int Hkv, const int32_t *page_ids, int num_pages_listed,
                            const void *k, uint8_t *thumb, uint8_t *resid, int *err,
                            cudaStream_t stream);
cudaError_t launch_append(int B, int Hkv, int P, int max_blocks, const int32_t *positions,
                          const int32_t *block_table, const void *k_new, const void *v_new,
                          uint8_t *thumb, uint8_t *resid, void *v_cache, void *k_cache, int *err,
                          cudaStream_t stream);
cudaError_t launch_decode(const DecodeArgs &a, int main_ctas, cudaStream_t stream);
cudaError_t launch_sparse(const DecodeArgs &a, int ctas, cudaStream_t stream);
cudaError_t launch_dense(const DecodeArgs &a, int ctas, cudaStream_t stream);
cudaError_t launch_select(const DecodeArgs &a, int selector, float budget, float *imp, float2 *ml,
                          cudaStream_t stream);
size_t select_smem_bytes(int max_blocks);
int select_max_blocks();
size_t art_list_bytes(int units, int max_blocks);
cudaError_t launch_art(const DecodeArgs &a, float tau, float phi, int patience, int32_t *used,
                       int32_t *list, cudaStream_t stream);
}  // namespace ffd

using namespace ffd;

namespace {

thread_local int g_last_cuda = 0;  // the cudaError_t behind this thread's latest FFD_ERR_CUDA

ffd_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return FFD_OK;
    g_last_cuda = static_cast<int>(e);
    return FFD_ERR_CUDA;
}

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// ART's workspace: the error word, then the units' traversal lists.
size_t art_workspace_bytes(const ffd_decode_params *p) {
    return kAlign + align_up(art_list_bytes(p->batch * p->num_kv_heads, p->max_blocks_per_seq));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Bound of every device wait of a call: the caller's, or the default.
uint64_t wait_bound_ns(const ffd_decode_params *p) {
    return p->wait_limit_us > 0 ? (uint64_t)p->wait_limit_us * 1000ull : kWaitTimeoutNs;
}

int current_sm_count() {
    static int cache[128];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e), -1;
    if (dev >= 0 && dev < 128 && cache[dev] > 0) return cache[dev];
    int v = 0;
    e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_status(e), -1;
    if (dev >= 0 && dev < 128) cache[dev] = v;
    return v;
}

ffd_status check_params(const ffd_decode_params *p) {
    if (!p) return FFD_ERR_INVALID_ARG;
    if (p->batch < 1 || p->num_q_heads < 1 || p->num_kv_heads < 1 || p->num_pages < 1 ||
        p->max_blocks_per_seq < 1 || p->sink_tokens < 0 || p->local_tokens < 0 ||
        p->num_splits < 0 || p->wait_limit_us < 0)
        return FFD_ERR_INVALID_ARG;
    if (p->schedule != FFD_SCHEDULE_FUSED && p->schedule != FFD_SCHEDULE_SCAN_REFINE)
        return FFD_ERR_INVALID_ARG;
    if (p->num_q_heads % p->num_kv_heads != 0) return FFD_ERR_INVALID_ARG;
    if (isnan(p->delta) || p->delta == -INFINITY) return FFD_ERR_INVALID_ARG;
    if (!isfinite(p->sm_scale) || !(p->sm_scale > 0.0f)) return FFD_ERR_INVALID_ARG;
    if (p->head_dim != kD || p->page_size != kPage) return FFD_ERR_UNSUPPORTED;
    const int G = p->num_q_heads / p->num_kv_heads;
    if (G < 1 || G > kMaxG) return FFD_ERR_UNSUPPORTED;
    // grid.y = B * Hkv, grid.x = splits / forced slots
    if ((int64_t)p->batch * p->num_kv_heads > 65535) return FFD_ERR_UNSUPPORTED;
    // the scan-then-refine kernel names a block by u * max_blocks_per_seq + block in an int32
    if (p->schedule == FFD_SCHEDULE_SCAN_REFINE &&
        (int64_t)p->batch * p->num_kv_heads * p->max_blocks_per_seq > INT32_MAX)
        return FFD_ERR_UNSUPPORTED;
    return FFD_OK;
}

// The library's CTA count (num_splits 0): one per SM, or fewer when the cache holds fewer than
// kMinBlocksPerCta blocks a CTA (B * Hkv * max_blocks_per_seq bounds the blocks from above, as the
// lengths are on the device): a tiny cache split over every SM pays the start-up of every CTA and
// the merge of as many records for a block or less each.
constexpr int64_t kMinBlocksPerCta = 4;
int default_ctas(const ffd_decode_params *p, int sms) {
    const int64_t blocks = (int64_t)p->batch * p->num_kv_heads * p->max_blocks_per_seq;
    const int64_t want = (blocks + kMinBlocksPerCta - 1) / kMinBlocksPerCta;
    return want < sms ? (want > 0 ? (int)want : 1) : sms;
}

struct Plan {
    int nf;    // stage-1 slots per unit (FFD step)
    int ctas;  // CTAs of the persistent kernel
    size_t m1_off, mt_off, part_off, kept_off, keptn_off, cnt_off, total;
};

// Split records per (unit, CTA): one per refine group, and the scan-then-refine kernel has three.
constexpr int kRecordGroups = 3;
// Per-unit counters: merge tickets, stage-1 slots, merge reports, merger declarations, and two
// buffers of kept-block counts (scan-then-refine); then the grid-barrier counter.
size_t counter_ints(size_t units) { return 6 * units + 1; }

// Workspace of ffd_decode_attention: [error word | stage-1 maxima | per-unit m~ | split records |
// kept-block lists | kept counts per CTA | counters]. Split records: one per (unit, CTA) pair that
// shares work and refine group, indexed (unit + cta) * groups + group. Stage 1 has one slot per
// forced block (at least one). The kept lists (one (unit, block) entry per block at most) and the
// per-CTA counts serve the scan-then-refine schedule.
ffd_status make_decode_plan(const ffd_decode_params *p, Plan *pl) {
    ffd_status st = check_params(p);
    if (st != FFD_OK) return st;
    const int64_t units = (int64_t)p->batch * p->num_kv_heads;
    const int G = p->num_q_heads / p->num_kv_heads;
    // one CTA per SM, all resident at once (the main kernel is a cooperative launch); without a
    // device to ask, an explicit count is taken as is (a size query then errs on the large side)
    const int sms = current_sm_count();
    int ctas = p->num_splits;
    if (ctas == 0) {
        if (sms <= 0) return FFD_ERR_CUDA;
        ctas = default_ctas(p, sms);
    } else if (sms > 0 && ctas > sms) {
        ctas = sms;
    }
    pl->ctas = ctas;
    const int nf = max_forced_blocks(p->sink_tokens, p->local_tokens, p->max_blocks_per_seq);
    pl->nf = nf > 0 ? nf : 1;
    size_t off = kAlign;
    pl->m1_off = off;
    off = align_up(off + (size_t)units * pl->nf * kMaxG * sizeof(float));
    pl->mt_off = off;
    off = align_up(off + (size_t)units * kMaxG * sizeof(float));
    pl->part_off = off;
    off = align_up(off + (size_t)(units + ctas) * kRecordGroups * G * kPartStride * sizeof(float));
    pl->kept_off = off;
    off = align_up(off + (size_t)units * p->max_blocks_per_seq * sizeof(int2));
    pl->keptn_off = off;
    off = align_up(off + (size_t)ctas * sizeof(int));
    pl->cnt_off = off;
    off = align_up(off + counter_ints(units) * sizeof(int));
    pl->total = off;
    return FFD_OK;
}

// Workspace of ffd_dense_decode: [error word | split records | counters], the FFD step's layout
// without the stage-1 parts (the dense kernel uses the same schedule, records and merge).
ffd_status make_dense_plan(const ffd_decode_params *p, Plan *pl) {
    ffd_status st = check_params(p);
    if (st != FFD_OK) return st;
    const int64_t units = (int64_t)p->batch * p->num_kv_heads;
    const int G = p->num_q_heads / p->num_kv_heads;
    const int sms = current_sm_count();
    int ctas = p->num_splits;
    if (ctas == 0) {
        if (sms <= 0) return FFD_ERR_CUDA;
        ctas = default_ctas(p, sms);
    } else if (sms > 0 && ctas > sms) {
        ctas = sms;
    }
    pl->ctas = ctas;
    pl->nf = 0;
    size_t off = kAlign;
    pl->m1_off = pl->mt_off = pl->kept_off = pl->keptn_off = off;
    pl->part_off = off;
    off = align_up(off + (size_t)(units + ctas) * kRefineGroups * G * kPartStride * sizeof(float));
    pl->cnt_off = off;
    off = align_up(off + 4 * (size_t)units * sizeof(int));
    pl->total = off;
    return FFD_OK;
}

cudaEvent_t g_prof_start = nullptr, g_prof_stop = nullptr;

DecodeArgs make_args(const ffd_decode_params *p, const Plan &pl, void *ws) {
    DecodeArgs a{};
    a.prof_start = g_prof_start;
    a.prof_stop = g_prof_stop;
    a.B = p->batch;
    a.Hq = p->num_q_heads;
    a.Hkv = p->num_kv_heads;
    a.G = p->num_q_heads / p->num_kv_heads;
    a.P = p->num_pages;
    a.max_blocks = p->max_blocks_per_seq;
    a.S = p->sink_tokens;
    a.L = p->local_tokens;
    a.nf = pl.nf;
    a.delta = p->delta;
    a.sm_scale = p->sm_scale;
    a.wait_ns = wait_bound_ns(p);
    char *base = static_cast<char *>(ws);
    a.err = reinterpret_cast<int *>(base);
    a.ws_m1 = reinterpret_cast<float *>(base + pl.m1_off);
    a.ws_mt = reinterpret_cast<float *>(base + pl.mt_off);
    a.ws_part = reinterpret_cast<float *>(base + pl.part_off);
    a.ws_kept = reinterpret_cast<int2 *>(base + pl.kept_off);
    a.ws_keptn = reinterpret_cast<int *>(base + pl.keptn_off);
    a.ws_cnt = reinterpret_cast<int *>(base + pl.cnt_off);
    const size_t units = (size_t)p->batch * p->num_kv_heads;
    a.ws_ukept = a.ws_cnt + 4 * units;
    a.ws_grid = reinterpret_cast<unsigned int *>(a.ws_cnt + 6 * units);
    return a;
}

}  // namespace

extern "C" {

int32_t ffd_last_cuda_error(void) { return g_last_cuda; }

int32_t ffd_suggest_schedule(int64_t total_blocks, int64_t kept_blocks) {
    if (total_blocks <= 0 || kept_blocks < 0 || kept_blocks > total_blocks)
        return FFD_SCHEDULE_FUSED;
    const int sms = current_sm_count();
    if (sms <= 0) return FFD_SCHEDULE_FUSED;
    // the scan-then-refine kernel reads the thumbnails once more than the fused one and gains by
    // scanning with every warp and balancing the refinement: that pays once the kept blocks are a
    // minority and every SM has a long enough scan
    return 2 * kept_blocks < total_blocks && total_blocks >= 64LL * sms ? FFD_SCHEDULE_SCAN_REFINE
                                                                      : FFD_SCHEDULE_FUSED;
}

const char *ffd_status_string(ffd_status s) {
    switch (s) {
        case FFD_OK: return "FFD_OK";
        case FFD_ERR_INVALID_ARG: return "FFD_ERR_INVALID_ARG";
        case FFD_ERR_UNSUPPORTED: return "FFD_ERR_UNSUPPORTED";
        case FFD_ERR_WORKSPACE: return "FFD_ERR_WORKSPACE";
        case FFD_ERR_CUDA: return "FFD_ERR_CUDA";
        case FFD_ERR_BOUNDS: return "FFD_ERR_BOUNDS";
        case FFD_ERR_RANGE: return "FFD_ERR_RANGE";
        case FFD_ERR_TIMEOUT: return "FFD_ERR_TIMEOUT";
    }
    return "FFD_ERR_UNKNOWN";
}

int32_t ffd_version(void) { return 300; }

ffd_status ffd_quantize_keys(const ffd_cache_desc *cache, const void *k_bf16, uint8_t *thumb,
                             uint8_t *resid, const int32_t *page_ids, int32_t num_page_ids,
                             int32_t *error_word, void *stream) {
    if (!cache || !k_bf16 || !thumb || !resid) return FFD_ERR_INVALID_ARG;
    if (cache->num_pages < 1 || cache->num_kv_heads < 1) return FFD_ERR_INVALID_ARG;
    if (page_ids && num_page_ids < 0) return FFD_ERR_INVALID_ARG;
    if (cache->head_dim != kD || cache->page_size != kPage) return FFD_ERR_UNSUPPORTED;
    if (!aligned16(k_bf16) || !aligned16(thumb) || !aligned16(resid)) return FFD_ERR_INVALID_ARG;
    const int listed = page_ids ? num_page_ids : cache->num_pages;
    if ((int64_t)listed * cache->num_kv_heads * kPage * 32 > INT32_MAX) return FFD_ERR_UNSUPPORTED;
    cudaError_t e = launch_quantize(cache->num_pages, cache->num_kv_heads, page_ids, listed, k_bf16,
                                    thumb, resid, error_word, static_cast<cudaStream_t>(stream));
    return cuda_status(e);
}

ffd_status ffd_append_kv(const ffd_cache_desc *cache, int32_t batch, int32_t max_blocks_per_seq,
                         const void *k_new_bf16, const void *v_new_bf16, const int32_t *positions,
                         const int32_t *block_table, uint8_t *thumb, uint8_t *resid,
                         void *v_bf16, void *k_bf16, int32_t *error_word, void *stream) {
    if (!cache || !k_new_bf16 || !v_new_bf16 || !positions || !block_table || !thumb || !resid ||
        !v_bf16)
        return FFD_ERR_INVALID_ARG;
    if (cache->num_pages < 1 || cache->num_kv_heads < 1 || batch < 1 || max_blocks_per_seq < 1)
        return FFD_ERR_INVALID_ARG;
    if (cache->head_dim != kD || cache->page_size != kPage) return FFD_ERR_UNSUPPORTED;
    if (!aligned16(k_new_bf16) || !aligned16(v_new_bf16) || !aligned16(thumb) ||
        !aligned16(resid) || !aligned16(v_bf16) || (k_bf16 && !aligned16(k_bf16)))
        return FFD_ERR_INVALID_ARG;
    if ((int64_t)batch * cache->num_kv_heads * 4 > INT32_MAX ||
        (int64_t)max_blocks_per_seq * kPage > INT32_MAX)
        return FFD_ERR_UNSUPPORTED;
    cudaError_t e = launch_append(batch, cache->num_kv_heads, cache->num_pages, max_blocks_per_seq,
                                  positions, block_table, k_new_bf16, v_new_bf16, thumb, resid,
                                  v_bf16, k_bf16, error_word, static_cast<cudaStream_t>(stream));
    return cuda_status(e);
}

size_t ffd_decode_workspace_size(const ffd_decode_params *params) {
    Plan pl;
    return make_decode_plan(params, &pl) == FFD_OK ? pl.total : 0;
}

size_t ffd_dense_workspace_size(const ffd_decode_params *params) {
    Plan pl;
    return make_dense_plan(params, &pl) == FFD_OK ? pl.total : 0;
}

ffd_status ffd_decode_attention(const ffd_decode_params *params, const void *q_bf16,
                                const uint8_t *thumb, const uint8_t *resid, const void *v_bf16,
                                const int32_t *seq_lens, const int32_t *block_table, float *out,
                                uint8_t *keep_mask, float *m_tilde, void *workspace,
                                size_t workspace_bytes, void *stream) {
    if (!q_bf16 || !thumb || !resid || !v_bf16 || !seq_lens || !block_table || !out || !workspace)
        return FFD_ERR_INVALID_ARG;
    if (!aligned16(thumb) || !aligned16(resid) || !aligned16(v_bf16) || !aligned16(q_bf16) ||
        (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)))
        return FFD_ERR_INVALID_ARG;
    Plan pl;
    ffd_status st = make_decode_plan(params, &pl);
    if (st != FFD_OK) return st;
    if (workspace_bytes < pl.total) return FFD_ERR_WORKSPACE;
    DecodeArgs a = make_args(params, pl, workspace);
    a.q = static_cast<const __nv_bfloat16 *>(q_bf16);
    a.thumb = thumb;
    a.resid = resid;
    a.v = static_cast<const __nv_bfloat16 *>(v_bf16);
    a.seq_lens = seq_lens;
    a.block_table = block_table;
    a.out = out;
    a.keep_mask = keep_mask;
    a.m_tilde = m_tilde;
    cudaError_t e = params->schedule == FFD_SCHEDULE_SCAN_REFINE
                        ? launch_sparse(a, pl.ctas, static_cast<cudaStream_t>(stream))
                        : launch_decode(a, pl.ctas, static_cast<cudaStream_t>(stream));
    return cuda_status(e);
}

ffd_status ffd_dense_decode(const ffd_decode_params *params, const void *q_bf16,
                            const void *k_bf16, const void *v_bf16, const int32_t *seq_lens,
                            const int32_t *block_table, float *out, void *workspace,
                            size_t workspace_bytes, void *stream) {
    if (!q_bf16 || !k_bf16 || !v_bf16 || !seq_lens || !block_table || !out || !workspace)
        return FFD_ERR_INVALID_ARG;
    if (!aligned16(k_bf16) || !aligned16(v_bf16) || !aligned16(q_bf16) ||
        (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)))
        return FFD_ERR_INVALID_ARG;
    Plan pl;
    ffd_status st = make_dense_plan(params, &pl);
    if (st != FFD_OK) return st;
    if (workspace_bytes < pl.total) return FFD_ERR_WORKSPACE;
    DecodeArgs a = make_args(params, pl, workspace);
    a.q = static_cast<const __nv_bfloat16 *>(q_bf16);
    a.k = static_cast<const __nv_bfloat16 *>(k_bf16);
    a.v = static_cast<const __nv_bfloat16 *>(v_bf16);
    a.seq_lens = seq_lens;
    a.block_table = block_table;
    a.out = out;
    cudaError_t e = launch_dense(a, pl.ctas, static_cast<cudaStream_t>(stream));
    return cuda_status(e);
}

// Workspace of ffd_select_blocks: [error word | importance [units][max_blocks] f32 |
// per-head (max, sum) [units][max_blocks][G] float2].
struct SelectPlan {
    size_t imp_off, ml_off, total;
};

ffd_status make_select_plan(const ffd_decode_params *p, SelectPlan *pl) {
    ffd_status st = check_params(p);
    if (st != FFD_OK) return st;
    if (p->max_blocks_per_seq > select_max_blocks()) return FFD_ERR_UNSUPPORTED;
    const size_t units = (size_t)p->batch * p->num_kv_heads;
    const size_t G = (size_t)(p->num_q_heads / p->num_kv_heads);
    pl->imp_off = kAlign;
    pl->ml_off = align_up(pl->imp_off + units * p->max_blocks_per_seq * sizeof(float));
    pl->total = align_up(pl->ml_off + units * p->max_blocks_per_seq * G * 2 * sizeof(float));
    return FFD_OK;
}

size_t ffd_select_workspace_size(const ffd_decode_params *params) {
    SelectPlan pl;
    return make_select_plan(params, &pl) == FFD_OK ? pl.total : 0;
}

ffd_status ffd_select_blocks(const ffd_decode_params *params, int32_t selector, float budget,
                             const void *q_bf16, const uint8_t *thumb, const int32_t *seq_lens,
                             const int32_t *block_table, uint8_t *keep_mask, void *workspace,
                             size_t workspace_bytes, void *stream) {
    if (!q_bf16 || !thumb || !seq_lens || !block_table || !keep_mask || !workspace)
        return FFD_ERR_INVALID_ARG;
    if (!aligned16(thumb) || !aligned16(q_bf16) ||
        (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)))
        return FFD_ERR_INVALID_ARG;
    if (selector == FFD_SELECT_TOPK) {
        if (!(budget >= 0.0f) || budget != floorf(budget) || budget > 2147483647.0f)
            return FFD_ERR_INVALID_ARG;
    } else if (selector == FFD_SELECT_TOPP) {
        if (!(budget > 0.0f && budget <= 1.0f)) return FFD_ERR_INVALID_ARG;
    } else {
        return FFD_ERR_INVALID_ARG;
    }
    SelectPlan pl;
    ffd_status st = make_select_plan(params, &pl);
    if (st != FFD_OK) return st;
    if (workspace_bytes < pl.total) return FFD_ERR_WORKSPACE;
    DecodeArgs a{};
    a.B = params->batch;
    a.Hq = params->num_q_heads;
    a.Hkv = params->num_kv_heads;
    a.G = params->num_q_heads / params->num_kv_heads;
    a.P = params->num_pages;
    a.max_blocks = params->max_blocks_per_seq;
    a.S = params->sink_tokens;
    a.L = params->local_tokens;
    a.sm_scale = params->sm_scale;
    a.wait_ns = wait_bound_ns(params);
    a.q = static_cast<const __nv_bfloat16 *>(q_bf16);
    a.thumb = thumb;
    a.seq_lens = seq_lens;
    a.block_table = block_table;
    a.keep_mask = keep_mask;
    char *base = static_cast<char *>(workspace);
    a.err = reinterpret_cast<int *>(base);
    cudaError_t e = launch_select(a, selector, budget, reinterpret_cast<float *>(base + pl.imp_off),
                                  reinterpret_cast<float2 *>(base + pl.ml_off),
                                  static_cast<cudaStream_t>(stream));
    return cuda_status(e);
}

ffd_status ffd_decode_attention_masked(const ffd_decode_params *params, const void *q_bf16,
                                       const uint8_t *thumb, const uint8_t *resid,
                                       const void *v_bf16, const int32_t *seq_lens,
                                       const int32_t *block_table, const uint8_t *keep_in,
                                       float *out, uint8_t *keep_mask, float *m_tilde,
                                       void *workspace, size_t workspace_bytes, void *stream) {
    if (!keep_in) return FFD_ERR_INVALID_ARG;
    if (!q_bf16 || !thumb || !resid || !v_bf16 || !seq_lens || !block_table || !out || !workspace)
        return FFD_ERR_INVALID_ARG;
    if (!aligned16(thumb) || !aligned16(resid) || !aligned16(v_bf16) || !aligned16(q_bf16) ||
        (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)))
        return FFD_ERR_INVALID_ARG;
    Plan pl;
    ffd_status st = make_decode_plan(params, &pl);
    if (st != FFD_OK) return st;
    if (workspace_bytes < pl.total) return FFD_ERR_WORKSPACE;
    DecodeArgs a = make_args(params, pl, workspace);
    a.q = static_cast<const __nv_bfloat16 *>(q_bf16);
    a.thumb = thumb;
    a.resid = resid;
    a.v = static_cast<const __nv_bfloat16 *>(v_bf16);
    a.seq_lens = seq_lens;
    a.block_table = block_table;
    a.out = out;
    a.keep_mask = keep_mask;
    a.keep_in = keep_in;
    a.m_tilde = m_tilde;
    cudaError_t e = launch_decode(a, pl.ctas, static_cast<cudaStream_t>(stream));
    return cuda_status(e);
}

// Workspace of ffd_art_attention: the error word only (the kernel keeps its state on chip).
size_t ffd_art_workspace_size(const ffd_decode_params *params) {
    return check_params(params) == FFD_OK ? art_workspace_bytes(params) : 0;
}

ffd_status ffd_art_attention(const ffd_decode_params *params, float tau, float phi,
                             int32_t patience, const void *q_bf16, const uint8_t *thumb,
                             const uint8_t *resid, const void *v_bf16, const int32_t *seq_lens,
                             const int32_t *block_table, const uint8_t *keep_in, float *out,
                             int32_t *blocks_used, void *workspace, size_t workspace_bytes,
                             void *stream) {
    if (!q_bf16 || !thumb || !resid || !v_bf16 || !seq_lens || !block_table || !out || !workspace)
        return FFD_ERR_INVALID_ARG;
    if (!aligned16(thumb) || !aligned16(resid) || !aligned16(v_bf16) || !aligned16(q_bf16) ||
        (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)))
        return FFD_ERR_INVALID_ARG;
    if (!(tau >= 0.0f) || !(phi >= 0.0f) || patience < 1) return FFD_ERR_INVALID_ARG;
    ffd_status st = check_params(params);
    if (st != FFD_OK) return st;
    if (workspace_bytes < art_workspace_bytes(params)) return FFD_ERR_WORKSPACE;
    DecodeArgs a{};
    a.B = params->batch;
    a.Hq = params->num_q_heads;
    a.Hkv = params->num_kv_heads;
    a.G = params->num_q_heads / params->num_kv_heads;
    a.P = params->num_pages;
    a.max_blocks = params->max_blocks_per_seq;
    a.sm_scale = params->sm_scale;
    a.wait_ns = wait_bound_ns(params);
    a.q = static_cast<const __nv_bfloat16 *>(q_bf16);
    a.thumb = thumb;
    a.resid = resid;
    a.v = static_cast<const __nv_bfloat16 *>(v_bf16);
    a.seq_lens = seq_lens;
    a.block_table = block_table;
    a.keep_in = keep_in;
    a.out = out;
    a.err = static_cast<int *>(workspace);
    cudaError_t e = launch_art(a, tau, phi, patience, blocks_used,
                               reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + kAlign),
                               static_cast<cudaStream_t>(stream));
    return cuda_status(e);
}

ffd_status ffd_set_profile_events(void *start, void *stop) {
    if ((start == nullptr) != (stop == nullptr)) return FFD_ERR_INVALID_ARG;
    g_prof_start = static_cast<cudaEvent_t>(start);
    g_prof_stop = static_cast<cudaEvent_t>(stop);
    return FFD_OK;
}

ffd_status ffd_get_error(void *error_word, void *stream) {
    if (!error_word) return FFD_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t h = 0;
    if (const cudaError_t e = cudaMemcpyAsync(&h, error_word, sizeof h, cudaMemcpyDeviceToHost, s);
        e != cudaSuccess)
        return cuda_status(e);
    if (const cudaError_t e = cudaStreamSynchronize(s); e != cudaSuccess) return cuda_status(e);
    if (h != 0) {
        cudaError_t e = cudaMemsetAsync(error_word, 0, sizeof h, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_status(e);
    }
    if (h & FFD_ERRBIT_BOUNDS) return FFD_ERR_BOUNDS;
    if (h & FFD_ERRBIT_RANGE) return FFD_ERR_RANGE;
    if (h & FFD_ERRBIT_TIMEOUT) return FFD_ERR_TIMEOUT;
    return FFD_OK;
}

// ---------------------------------------------------------------------------------------------
// Allocation-free decode: the same kernels, with their scratch in a fixed static device array.
//
// Some callers cannot hand the library a workspace: a plain C host that links only libffd.so and
// owns no device allocator, or a serving process that has carved all device memory into its
// KV-cache pool up front and may not allocate (cudaMalloc can also synchronise the device, which
// a latency-critical decode loop must avoid). For them the scratch lives in the array below,
// which every GPU that loads this library holds until the process exits.
// ---------------------------------------------------------------------------------------------
}  // extern "C"

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
void *g_static_ptr[kMaxDevices];
void *g_static_ctx[kMaxDevices];  // the context g_static_ptr[dev] was looked up in

// The CUDA context current on this thread (null before the runtime has made one). A
// cudaDeviceReset replaces the device's primary context, and the module's symbol addresses go
// with it.
void *current_context() {
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    }
    CUcontext c = nullptr;
    if (fn && fn(&c) != CUDA_SUCCESS) c = nullptr;
    return c;
}

// Device address of g_static_scratch on the current device (host code must not use the array's
// name as an address). Looked up with that device current, again whenever the current context is
// not the one of the last look-up (after a cudaDeviceReset, say).
ffd_status static_scratch(void **out) {
    int dev = 0;
    if (const cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= kMaxDevices) return FFD_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_static_mu);
    void *ctx = current_context();
    if (!g_static_ptr[dev] || !ctx || ctx != g_static_ctx[dev]) {
        void *p = nullptr;  // the look-up makes the primary context if there is none yet
        if (const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch); e != cudaSuccess)
            return cuda_status(e);
        if (!p) return FFD_ERR_CUDA;
        g_static_ptr[dev] = p;
        g_static_ctx[dev] = current_context();
    }
    *out = g_static_ptr[dev];
    return FFD_OK;
}

}  // namespace

extern "C" {

ffd_status ffd_decode_attention_static(const ffd_decode_params *params, const void *q_bf16,
                                       const uint8_t *thumb, const uint8_t *resid,
                                       const void *v_bf16, const int32_t *seq_lens,
                                       const int32_t *block_table, float *out,
                                       uint8_t *keep_mask, float *m_tilde, int32_t *error_word,
                                       void *stream) {
    if (!q_bf16 || !thumb || !resid || !v_bf16 || !seq_lens || !block_table || !out)
        return FFD_ERR_INVALID_ARG;
    if (!aligned16(thumb) || !aligned16(resid) || !aligned16(v_bf16) || !aligned16(q_bf16))
        return FFD_ERR_INVALID_ARG;
    Plan pl;
    ffd_status st = make_decode_plan(params, &pl);
    if (st != FFD_OK) return st;
    if (pl.total > kStaticScratchBytes) return FFD_ERR_WORKSPACE;
    void *ws = nullptr;
    st = static_scratch(&ws);
    if (st != FFD_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents: the error word and the per-unit tickets of
    // the in-kernel merge must start at zero.
    const size_t units = (size_t)params->batch * params->num_kv_heads;
    cudaError_t e = cudaMemsetAsync(ws, 0, kAlign, s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(static_cast<char *>(ws) + pl.cnt_off, 0,
                            counter_ints(units) * sizeof(int), s);
    if (e != cudaSuccess) return cuda_status(e);
    DecodeArgs a = make_args(params, pl, ws);
    if (error_word) a.err = reinterpret_cast<int *>(error_word);
    a.q = static_cast<const __nv_bfloat16 *>(q_bf16);
    a.thumb = thumb;
    a.resid = resid;
    a.v = static_cast<const __nv_bfloat16 *>(v_bf16);
    a.seq_lens = seq_lens;
    a.block_table = block_table;
    a.out = out;
    a.keep_mask = keep_mask;
    a.m_tilde = m_tilde;
    e = params->schedule == FFD_SCHEDULE_SCAN_REFINE ? launch_sparse(a, pl.ctas, s)
                                                     : launch_decode(a, pl.ctas, s);
    return cuda_status(e);
}

}  // extern "C"
