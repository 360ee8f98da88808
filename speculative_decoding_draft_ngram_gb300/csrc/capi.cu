// C ABI of libspecng: argument checks, workspace layout, the device status
// word and the launches.  Declarations and documentation: include/specng.h.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include "kv.cuh"
#include "ngram.cuh"
#include "verify.cuh"

namespace specng {

__device__ unsigned g_status_word;

// Diagnostic counters of the rarely taken exact paths (SPECNG_DIAG_*).
__device__ unsigned g_diag_counters[SPECNG_DIAG_N];

// Scratch of spec_verify_noalloc: part of the library's device image, one
// per device, so that callers without an allocator (see the header) can
// verify.  Each call zero-fills the part it uses before its kernels run.
static __device__ __align__(256) unsigned char g_verify_scratch[SPECNG_STATIC_SCRATCH_BYTES];

namespace {

thread_local char g_last_error[256] = "";

int fail(int code, const char* what) {
    std::snprintf(g_last_error, sizeof(g_last_error), "%s", what);
    return code;
}

int fail_cuda(cudaError_t e, const char* where) {
    std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", where, cudaGetErrorString(e));
    return SPECNG_ECUDA;
}

// Device address of the status word, looked up once per device.
unsigned* status_ptr() {
    static std::mutex mu;
    static unsigned* ptrs[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (ptrs[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) == cudaSuccess) ptrs[dev] = static_cast<unsigned*>(p);
    }
    return ptrs[dev];
}

// Device address of the diagnostic counters, looked up once per device.
unsigned* diag_ptr() {
    static std::mutex mu;
    static unsigned* ptrs[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (ptrs[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_diag_counters) == cudaSuccess) ptrs[dev] = static_cast<unsigned*>(p);
    }
    return ptrs[dev];
}

// The stream must belong to the current device: the status word, the
// counters and the static scratch are looked up on the current device.
bool stream_on_current_device(cudaStream_t s) {
    if (s == nullptr) return true;  // the legacy default stream follows the current device
    // a stream being captured into a graph takes no device query (it would end the
    // capture); a launch on another device's stream fails the capture by itself
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (cs != cudaStreamCaptureStatusNone) return true;
    int cur = -1, sd = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return false;
    if (cudaStreamGetDevice(s, &sd) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return cur == sd;
}

// Device address of the static verify scratch, looked up once per device
// (the lookup may load the module, so it belongs to set-up, before capture).
void* static_scratch_ptr() {
    static std::mutex mu;
    static void* ptrs[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (ptrs[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_verify_scratch) == cudaSuccess) ptrs[dev] = p;
    }
    return ptrs[dev];
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
    size_t part, bmax, blkws, rowres, seqres, part2, tickets, total;
    size_t row_thr, seq_ticket2;
    size_t row_tix, seq_state, ema_new, cool_new, grid_tix;
};

// The f32 chunks are the smaller ones, so their counts bound both dtypes.
int max_chunks(int V) { return (V + chunk_elems<false>() - 1) / chunk_elems<false>(); }
int max_chunks2(int V) { return (V + res_chunk_elems<false>() - 1) / res_chunk_elems<false>(); }

// per_block: one sum record per row and noise block (the fused LM-head path)
WsLayout ws_layout(int B, int K, int V, bool per_block = false) {
    const size_t rows = static_cast<size_t>(B) * (K + 1);
    const size_t nch = static_cast<size_t>(per_block ? noise_blocks(V) : max_chunks(V));
    const size_t nblk = static_cast<size_t>(noise_blocks(V));
    WsLayout L{};
    size_t off = 0;
    L.part = off;    off = align256(off + rows * nch * sizeof(SegSum));
    L.bmax = off;    off = align256(off + rows * nblk * sizeof(float));
    L.blkws = off;
    if (nblk > static_cast<size_t>(kSmemBlkCap)) off = align256(off + static_cast<size_t>(B) * nblk * kBlkScratchBytes);
    L.rowres = off;  off = align256(off + rows * sizeof(RowRes));
    L.seqres = off;  off = align256(off + static_cast<size_t>(B) * sizeof(SeqRes));
    L.part2 = off;   off = align256(off + static_cast<size_t>(B) * static_cast<size_t>(max_chunks2(V)) * sizeof(Partial));
    L.row_tix = off;    off = align256(off + rows * sizeof(unsigned long long));
    L.seq_state = off;  off = align256(off + static_cast<size_t>(B) * sizeof(unsigned long long));
    L.ema_new = off;    off = align256(off + static_cast<size_t>(B) * sizeof(float));
    L.cool_new = off;   off = align256(off + static_cast<size_t>(B) * sizeof(int32_t));
    L.tickets = off;
    L.row_thr = off;      off += rows * sizeof(unsigned);
    L.seq_ticket2 = off;  off += static_cast<size_t>(B) * sizeof(unsigned);
    L.grid_tix = off;     off += sizeof(unsigned);
    L.total = align256(off);
    return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tag of one verify call, in [1, 2^31): the single-kernel schedule's tickets
// and state words carry it, so words left by earlier calls read as empty and
// nothing needs clearing between calls.
uint32_t next_epoch() {
    static std::atomic<uint32_t> counter{0};
    uint32_t e = 0;
    while (e == 0) e = (counter.fetch_add(1u) + 1u) & 0x7FFFFFFFu;
    return e;
}

}  // namespace
}  // namespace specng

using namespace specng;

struct specng_ngram {
    NgramDev dev;
    void* mem;
    int grid;
};

extern "C" {

const char* specng_last_error(void) { return g_last_error; }

const char* specng_strerror(int code) {
    switch (code) {
        case SPECNG_OK: return "ok";
        case SPECNG_EINVAL: return "invalid argument (null pointer, size or parameter out of range)";
        case SPECNG_EALIGN: return "pointer alignment below what the call requires";
        case SPECNG_ECUDA: return "CUDA runtime error";
        case SPECNG_ENOMEM: return "device allocation failed";
        case SPECNG_ESMALL: return "workspace smaller than spec_verify_workspace_bytes";
        default: return "unknown error code";
    }
}

int specng_set_verify_marker(cudaEvent_t after_stream_kernel) {
    verify_marker() = after_stream_kernel;
    return SPECNG_OK;
}

namespace {

int kv_view(const specng_kv_pool* pool, const char* what, specng::KvDev* out) {
    if (pool == nullptr || pool->free_stack == nullptr || pool->free_top == nullptr || pool->block_table == nullptr ||
        pool->nblocks == nullptr) {
        std::snprintf(g_last_error, sizeof(g_last_error), "%s: NULL pool or pool array", what);
        return SPECNG_EINVAL;
    }
    if (pool->num_blocks < 1 || pool->num_blocks > (1 << 30) || pool->B < 1 || pool->B > (1 << 20) ||
        pool->max_blocks < 1 || pool->block_size < 1 ||
        static_cast<int64_t>(pool->B) * pool->max_blocks > 0x7FFFFFFFLL) {
        std::snprintf(g_last_error, sizeof(g_last_error), "%s: pool sizes out of range", what);
        return SPECNG_EINVAL;
    }
    out->free_stack = pool->free_stack;
    out->free_top = pool->free_top;
    out->table = pool->block_table;
    out->nblocks = pool->nblocks;
    out->num_blocks = pool->num_blocks;
    out->B = pool->B;
    out->max_blocks = pool->max_blocks;
    out->block_size = pool->block_size;
    out->status = status_ptr();
    return SPECNG_OK;
}

}  // namespace

int specng_kv_init(const specng_kv_pool* pool, cudaStream_t s) {
    specng::KvDev K;
    const int rc = kv_view(pool, "specng_kv_init", &K);
    if (rc != SPECNG_OK) return rc;
    const cudaError_t e = launch_kv_init(K, s);
    return e == cudaSuccess ? SPECNG_OK : fail_cuda(e, "specng_kv_init");
}

int specng_kv_reserve(const specng_kv_pool* pool, const int32_t* kv_len, int extra, cudaStream_t s) {
    specng::KvDev K;
    const int rc = kv_view(pool, "specng_kv_reserve", &K);
    if (rc != SPECNG_OK) return rc;
    if (kv_len == nullptr || extra < 0) return fail(SPECNG_EINVAL, "specng_kv_reserve: NULL kv_len or extra < 0");
    const cudaError_t e = launch_kv_reserve(K, kv_len, extra, s);
    return e == cudaSuccess ? SPECNG_OK : fail_cuda(e, "specng_kv_reserve");
}

int specng_kv_trim(const specng_kv_pool* pool, const int32_t* kv_len, cudaStream_t s) {
    specng::KvDev K;
    const int rc = kv_view(pool, "specng_kv_trim", &K);
    if (rc != SPECNG_OK) return rc;
    if (kv_len == nullptr) return fail(SPECNG_EINVAL, "specng_kv_trim: NULL kv_len");
    const cudaError_t e = launch_kv_trim(K, kv_len, s);
    return e == cudaSuccess ? SPECNG_OK : fail_cuda(e, "specng_kv_trim");
}

int specng_kv_release(const specng_kv_pool* pool, const int32_t* done, cudaStream_t s) {
    specng::KvDev K;
    const int rc = kv_view(pool, "specng_kv_release", &K);
    if (rc != SPECNG_OK) return rc;
    if (done == nullptr) return fail(SPECNG_EINVAL, "specng_kv_release: NULL done");
    const cudaError_t e = launch_kv_release(K, done, s);
    return e == cudaSuccess ? SPECNG_OK : fail_cuda(e, "specng_kv_release");
}

int specng_step_advance(uint64_t* step_dev, cudaStream_t s) {
    if (step_dev == nullptr) return fail(SPECNG_EINVAL, "specng_step_advance: NULL step_dev");
    const cudaError_t e = launch_step_advance(step_dev, s);
    return e == cudaSuccess ? SPECNG_OK : fail_cuda(e, "specng_step_advance");
}

int specng_get_status(uint32_t* bits, int clear) {
    if (bits == nullptr) return fail(SPECNG_EINVAL, "specng_get_status: bits is NULL");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda(e, "specng_get_status");
    unsigned v = 0;
    e = cudaMemcpyFromSymbol(&v, g_status_word, sizeof(v));
    if (e != cudaSuccess) return fail_cuda(e, "specng_get_status");
    *bits = v;
    if (clear) {
        const unsigned z = 0;
        e = cudaMemcpyToSymbol(g_status_word, &z, sizeof(z));
        if (e != cudaSuccess) return fail_cuda(e, "specng_get_status");
    }
    return SPECNG_OK;
}

// ------------------------------------------------------------------ n-gram

int specng_ngram_create(specng_ngram** table, int B, int V, int64_t max_positions, cudaStream_t s) {
    if (table == nullptr) return fail(SPECNG_EINVAL, "specng_ngram_create: table is NULL");
    *table = nullptr;
    if (B < 1 || B > SPECNG_NGRAM_MAX_B) return fail(SPECNG_EINVAL, "specng_ngram_create: B outside [1, 512]");
    if (V < 1 || V > SPECNG_NGRAM_MAX_V) return fail(SPECNG_EINVAL, "specng_ngram_create: V outside [1, 2^18]");
    if (max_positions < 1 || max_positions > (int64_t(1) << 33))
        return fail(SPECNG_EINVAL, "specng_ngram_create: max_positions outside [1, 2^33]");
    uint64_t slots = 1024;
    while (slots < 2ull * static_cast<uint64_t>(max_positions)) slots <<= 1;
    const size_t table_bytes = slots * sizeof(ulonglong2);
    const size_t idx_bytes = align256(2 * static_cast<size_t>(B) * sizeof(int32_t));
    void* mem = nullptr;
    cudaError_t e = cudaMalloc(&mem, 4 * table_bytes + idx_bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SPECNG_ENOMEM, "specng_ngram_create: cudaMalloc failed");
    }
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    specng_ngram* t = new specng_ngram();
    char* base = static_cast<char*>(mem);
    t->mem = mem;
    t->grid = 2 * (sms > 0 ? sms : 1);
    t->dev.tri_pair = reinterpret_cast<ulonglong2*>(base);
    t->dev.bi_pair = reinterpret_cast<ulonglong2*>(base + table_bytes);
    t->dev.tri_ctx = reinterpret_cast<ulonglong2*>(base + 2 * table_bytes);
    t->dev.bi_ctx = reinterpret_cast<ulonglong2*>(base + 3 * table_bytes);
    t->dev.mask = slots - 1;
    t->dev.indexed[0] = reinterpret_cast<int32_t*>(base + 4 * table_bytes);
    t->dev.indexed[1] = t->dev.indexed[0] + B;
    t->dev.B = B;
    t->dev.V = V;
    t->dev.status = status_ptr();
    t->dev.min_count = 1;
    e = launch_ngram_clear(t->dev, s);
    if (e != cudaSuccess) {
        cudaFree(mem);
        delete t;
        return fail_cuda(e, "specng_ngram_create");
    }
    *table = t;
    return SPECNG_OK;
}

int specng_ngram_destroy(specng_ngram* table) {
    if (table == nullptr) return SPECNG_OK;
    cudaError_t e = cudaDeviceSynchronize();
    cudaError_t f = cudaFree(table->mem);
    delete table;
    if (e != cudaSuccess) return fail_cuda(e, "specng_ngram_destroy");
    if (f != cudaSuccess) return fail_cuda(f, "specng_ngram_destroy");
    return SPECNG_OK;
}

int specng_ngram_reset(specng_ngram* table, cudaStream_t s) {
    if (table == nullptr) return fail(SPECNG_EINVAL, "specng_ngram_reset: table is NULL");
    const cudaError_t e = launch_ngram_clear(table->dev, s);
    if (e != cudaSuccess) return fail_cuda(e, "specng_ngram_reset");
    return SPECNG_OK;
}

int specng_ngram_set_min_count(specng_ngram* table, int min_count) {
    if (table == nullptr) return fail(SPECNG_EINVAL, "specng_ngram_set_min_count: table is NULL");
    if (min_count < 1 || min_count > (1 << 22) - 1)
        return fail(SPECNG_EINVAL, "specng_ngram_set_min_count: min_count outside [1, 2^22 - 1]");
    table->dev.min_count = static_cast<uint64_t>(min_count);
    return SPECNG_OK;
}

int specng_ngram_capacity(const specng_ngram* table, int64_t* slots) {
    if (table == nullptr || slots == nullptr) return fail(SPECNG_EINVAL, "specng_ngram_capacity: NULL argument");
    *slots = static_cast<int64_t>(table->dev.mask + 1);
    return SPECNG_OK;
}

int ngram_update(const int32_t* history, int64_t hist_stride, const int32_t* lens, specng_ngram* table,
                 cudaStream_t s) {
    if (table == nullptr || history == nullptr || lens == nullptr)
        return fail(SPECNG_EINVAL, "ngram_update: NULL argument");
    if (hist_stride < 1 || hist_stride > SPECNG_NGRAM_MAX_POS)
        return fail(SPECNG_EINVAL, "ngram_update: hist_stride outside [1, 2^24]");
    const cudaError_t e = launch_ngram_update(table->dev, history, hist_stride, lens, table->grid, s);
    if (e != cudaSuccess) return fail_cuda(e, "ngram_update");
    return SPECNG_OK;
}

int ngram_draft(const specng_ngram* table, const int32_t* history, int64_t hist_stride, const int32_t* lens,
                int max_k, const int32_t* k_limit, const int32_t* fallback, int32_t* out_drafts, int32_t* out_k,
                cudaStream_t s) {
    if (table == nullptr || history == nullptr || lens == nullptr || out_k == nullptr)
        return fail(SPECNG_EINVAL, "ngram_draft: NULL argument");
    if (max_k < 0 || max_k > SPECNG_MAX_K) return fail(SPECNG_EINVAL, "ngram_draft: max_k outside [0, 16]");
    if (max_k > 0 && out_drafts == nullptr) return fail(SPECNG_EINVAL, "ngram_draft: out_drafts is NULL");
    if (hist_stride < 1 || hist_stride > SPECNG_NGRAM_MAX_POS)
        return fail(SPECNG_EINVAL, "ngram_draft: hist_stride outside [1, 2^24]");
    const cudaError_t e = launch_ngram_draft(table->dev, history, hist_stride, lens, max_k, k_limit, fallback,
                                             out_drafts, out_k, s);
    if (e != cudaSuccess) return fail_cuda(e, "ngram_draft");
    return SPECNG_OK;
}

// ------------------------------------------------------------------ verify

size_t spec_verify_workspace_bytes(int B, int K, int V) {
    if (B < 1 || K < 0 || K > SPECNG_MAX_K || V < 1) return 0;
    return ws_layout(B, K, V).total;
}

int spec_verify_workspace_init(void* workspace, size_t workspace_bytes, cudaStream_t s) {
    if (workspace == nullptr) return fail(SPECNG_EINVAL, "spec_verify_workspace_init: workspace is NULL");
    const cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes, s);
    if (e != cudaSuccess) return fail_cuda(e, "spec_verify_workspace_init");
    return SPECNG_OK;
}

namespace {

// Host-side checks of a verify call and its kernel parameters, everything
// but the workspace.  Nothing is enqueued here.
int verify_setup(const char* who, const void* logits, int logits_dtype, int B, int K, int V, const int32_t* drafts,
                 const float* draft_probs, const int32_t* k, const int32_t* history, int64_t hist_stride,
                 const int32_t* lens, const specng_verify_params* params, int32_t* kv_len, float* ema,
                 int32_t* out_tokens, int32_t* out_accept_len, cudaStream_t s, VerifyDev* out, bool* flags) {
    char msg[160];
    auto bad = [&](int code, const char* what) {
        std::snprintf(msg, sizeof(msg), "%s: %s", who, what);
        return fail(code, msg);
    };
    if (logits == nullptr || k == nullptr || params == nullptr || kv_len == nullptr || ema == nullptr ||
        out_tokens == nullptr || out_accept_len == nullptr)
        return bad(SPECNG_EINVAL, "NULL argument");
    if (logits_dtype != SPECNG_BF16 && logits_dtype != SPECNG_F32)
        return bad(SPECNG_EINVAL, "logits_dtype must be SPECNG_BF16 or SPECNG_F32");
    if (B < 1 || B > (1 << 20)) return bad(SPECNG_EINVAL, "B outside [1, 2^20]");
    if (K < 0 || K > SPECNG_MAX_K) return bad(SPECNG_EINVAL, "K outside [0, 16]");
    if (V < 1 || V > (1 << 30)) return bad(SPECNG_EINVAL, "V outside [1, 2^30]");
    if (K > 0 && drafts == nullptr) return bad(SPECNG_EINVAL, "drafts is NULL with K > 0");
    const specng_verify_params& p = *params;
    if (!(p.temperature >= 0.0f) || !std::isfinite(p.temperature))
        return bad(SPECNG_EINVAL, "temperature must be finite and >= 0");
    if (!std::isfinite(p.softcap)) return bad(SPECNG_EINVAL, "softcap must be finite");
    if (!(p.rep_penalty > 0.0f) || !std::isfinite(p.rep_penalty))
        return bad(SPECNG_EINVAL, "rep_penalty must be finite and > 0");
    if (p.rep_window < 0 || p.rep_window > SPECNG_MAX_REP_WINDOW) return bad(SPECNG_EINVAL, "rep_window outside [0, 256]");
    if (p.gate_enabled && (!std::isfinite(p.ema_tau) || !std::isfinite(p.ema_thresh)))
        return bad(SPECNG_EINVAL, "ema_tau and ema_thresh must be finite");
    if (p.schedule < SPECNG_SCHEDULE_AUTO || p.schedule > SPECNG_SCHEDULE_SPLIT)
        return bad(SPECNG_EINVAL, "schedule must be SPECNG_SCHEDULE_AUTO, _FUSED or _SPLIT");
    if (p.schedule == SPECNG_SCHEDULE_FUSED && B > SPECNG_FUSED_MAX_B)
        return bad(SPECNG_EINVAL, "the single-kernel schedule takes B <= 2048");
    if (p.early_exit != 0 && p.early_exit != 1) return bad(SPECNG_EINVAL, "early_exit must be 0 or 1");
    if (p.probe_interval < 0) return bad(SPECNG_EINVAL, "probe_interval must be >= 0");
    if (p.cool_steps < 0) return bad(SPECNG_EINVAL, "cool_steps must be >= 0");
    if (p.cool_steps > 0 && p.gate_state == nullptr) return bad(SPECNG_EINVAL, "cool_steps > 0 needs gate_state");
    if (p.step_dev != nullptr && p.schedule == SPECNG_SCHEDULE_FUSED)
        return bad(SPECNG_EINVAL, "step_dev is not supported by the single-kernel schedule (per-call state tags)");
    const bool penalty = p.rep_penalty != 1.0f && p.rep_window > 0;
    if (penalty && (history == nullptr || lens == nullptr || hist_stride < 1))
        return bad(SPECNG_EINVAL, "history, lens and hist_stride are needed for the penalty");
    if (!stream_on_current_device(s))
        return bad(SPECNG_EINVAL, "the stream does not belong to the current device (make its device current)");
    const bool bf16 = logits_dtype == SPECNG_BF16;
    const int chunk = bf16 ? chunk_elems<true>() : chunk_elems<false>();
    const int nchunk = (V + chunk - 1) / chunk;
    const int chunk2 = bf16 ? res_chunk_elems<true>() : res_chunk_elems<false>();
    const int nchunk2 = (V + chunk2 - 1) / chunk2;
    if (static_cast<int64_t>(B) * (K + 1) * nchunk2 > 0x7FFFFFFFLL)
        return bad(SPECNG_EINVAL, "B * (K + 1) * chunks exceeds the grid limit");

    const bool greedy = p.temperature == 0.0f;
    const bool softcap = p.softcap > 0.0f;
    const bool dense = draft_probs != nullptr;
    const int epv = bf16 ? 8 : 4;

    VerifyDev& P = *out;
    P = VerifyDev{};
    P.logits = logits;
    P.B = B; P.K = K; P.V = V; P.nchunk = nchunk; P.nchunk2 = nchunk2;
    P.nblk = noise_blocks(V);
    P.drafts = drafts; P.q = draft_probs; P.k = k;
    P.hist = history; P.hist_stride = hist_stride; P.lens = lens;
    P.T = p.temperature;
    P.invT = greedy ? 0.0f : 1.0f / p.temperature;
    P.sc = greedy ? 0.0f : kLog2e / p.temperature;
    P.Td = static_cast<double>(p.temperature);
    P.cap = softcap ? p.softcap : 0.0f;
    P.invcap = softcap ? 1.0f / p.softcap : 0.0f;
    P.cap2l = softcap ? 2.0f * kLog2e / p.softcap : 0.0f;
    P.rep = p.rep_penalty;
    P.invrep = 1.0f / p.rep_penalty;
    P.W = penalty ? p.rep_window : 0;
    P.tau = p.ema_tau;
    P.thresh = p.ema_thresh;
    P.gate = p.gate_enabled ? 1 : 0;
    P.nk.k0 = static_cast<uint32_t>(p.seed);
    P.nk.k1 = static_cast<uint32_t>(p.seed >> 32);
    P.nk.step = static_cast<uint32_t>(p.step);
    P.probe = p.probe_interval;
    P.step64 = p.step;
    P.step_dev = p.step_dev;
    P.cool = p.cool_steps;
    P.gate_state = p.cool_steps > 0 ? p.gate_state : nullptr;
    P.nk.seq = 0;
    P.aligned = aligned16(logits) && (V % epv == 0) && (!dense || (aligned16(draft_probs) && V % 4 == 0));
    P.kv_len = kv_len; P.ema = ema; P.out_tokens = out_tokens; P.out_accept = out_accept_len;
    P.status = status_ptr();
    P.diag = diag_ptr();
    P.fused = p.schedule == SPECNG_SCHEDULE_FUSED ? 1 : 0;
    P.early_exit = P.fused ? p.early_exit : 0;
    P.epoch = next_epoch();
    flags[0] = bf16; flags[1] = greedy; flags[2] = softcap; flags[3] = penalty; flags[4] = dense;
    return SPECNG_OK;
}

void attach_workspace(VerifyDev& P, void* workspace, bool per_block = false) {
    const WsLayout L = ws_layout(P.B, P.K, P.V, per_block);
    char* ws = static_cast<char*>(workspace);
    P.part = reinterpret_cast<SegSum*>(ws + L.part);
    P.bmax = reinterpret_cast<float*>(ws + L.bmax);
    P.blkws = reinterpret_cast<uint8_t*>(ws + L.blkws);
    P.rowres = reinterpret_cast<RowRes*>(ws + L.rowres);
    P.seqres = reinterpret_cast<SeqRes*>(ws + L.seqres);
    P.part2 = reinterpret_cast<Partial*>(ws + L.part2);
    P.row_thr = reinterpret_cast<unsigned*>(ws + L.row_thr);
    P.seq_ticket2 = reinterpret_cast<unsigned*>(ws + L.seq_ticket2);
    P.row_tix = reinterpret_cast<unsigned long long*>(ws + L.row_tix);
    P.seq_state = reinterpret_cast<unsigned long long*>(ws + L.seq_state);
    P.ema_new = reinterpret_cast<float*>(ws + L.ema_new);
    P.cool_new = reinterpret_cast<int32_t*>(ws + L.cool_new);
    P.grid_tix = reinterpret_cast<unsigned*>(ws + L.grid_tix);
}

int verify_launch(const VerifyDev& P, const bool* f, cudaStream_t s, const char* who) {
    const cudaError_t e = f[0] ? launch_verify_dtype<true>(P, f[1], f[2], f[3], f[4], s)
                               : launch_verify_dtype<false>(P, f[1], f[2], f[3], f[4], s);
    if (e != cudaSuccess) return fail_cuda(e, who);
    return SPECNG_OK;
}

}  // namespace

int spec_verify(const void* logits, int logits_dtype, int B, int K, int V, const int32_t* drafts,
                const float* draft_probs, const int32_t* k, const int32_t* history, int64_t hist_stride,
                const int32_t* lens, const specng_verify_params* params, int32_t* kv_len, float* ema,
                int32_t* out_tokens, int32_t* out_accept_len, void* workspace, size_t workspace_bytes,
                cudaStream_t s) {
    VerifyDev P;
    bool f[5];
    int rc = verify_setup("spec_verify", logits, logits_dtype, B, K, V, drafts, draft_probs, k, history, hist_stride,
                          lens, params, kv_len, ema, out_tokens, out_accept_len, s, &P, f);
    if (rc != SPECNG_OK) return rc;
    if (workspace == nullptr) return fail(SPECNG_EINVAL, "spec_verify: workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(SPECNG_EALIGN, "spec_verify: workspace must be 256-byte aligned");
    if (workspace_bytes < ws_layout(B, K, V).total) return fail(SPECNG_ESMALL, "spec_verify: workspace too small");
    attach_workspace(P, workspace);
    return verify_launch(P, f, s, "spec_verify");
}

size_t spec_verify_lmhead_workspace_bytes(int B, int K, int V) {
    if (B < 1 || K < 0 || K > SPECNG_MAX_K || V < 1) return 0;
    return ws_layout(B, K, V, true).total;
}

int spec_verify_lmhead(const void* hidden, const void* weight, int d, void* logits, int B, int K, int V,
                       const int32_t* drafts, const float* draft_probs, const int32_t* k, const int32_t* history,
                       int64_t hist_stride, const int32_t* lens, const specng_verify_params* params, int32_t* kv_len,
                       float* ema, int32_t* out_tokens, int32_t* out_accept_len, void* workspace,
                       size_t workspace_bytes, cudaStream_t s) {
    const char* who = "spec_verify_lmhead";
    char msg[160];
    auto bad = [&](int code, const char* what) {
        std::snprintf(msg, sizeof(msg), "%s: %s", who, what);
        return fail(code, msg);
    };
    if (hidden == nullptr || weight == nullptr || logits == nullptr) return bad(SPECNG_EINVAL, "NULL argument");
    if (!aligned16(hidden) || !aligned16(weight) || !aligned16(logits))
        return bad(SPECNG_EALIGN, "hidden, weight and logits must be 16-byte aligned");
    if (d < 64 || d % 64 != 0 || d > (1 << 20)) return bad(SPECNG_EINVAL, "d must be a multiple of 64 in [64, 2^20]");
    if (V % 8 != 0) return bad(SPECNG_EINVAL, "V must be a multiple of 8");
    if (params != nullptr && params->rep_penalty != 1.0f && params->rep_window > 0)
        return bad(SPECNG_EINVAL, "the repetition penalty is not supported by the fused LM-head path");
    if (params != nullptr && params->schedule == SPECNG_SCHEDULE_FUSED)
        return bad(SPECNG_EINVAL, "the fused LM-head path runs the split schedule's decision kernel");
    VerifyDev P;
    bool f[5];
    int rc = verify_setup(who, logits, SPECNG_BF16, B, K, V, drafts, draft_probs, k, history, hist_stride, lens, params,
                          kv_len, ema, out_tokens, out_accept_len, s, &P, f);
    if (rc != SPECNG_OK) return rc;
    if (workspace == nullptr) return bad(SPECNG_EINVAL, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return bad(SPECNG_EALIGN, "workspace must be 256-byte aligned");
    if (workspace_bytes < ws_layout(B, K, V, true).total) return bad(SPECNG_ESMALL, "workspace too small");
    attach_workspace(P, workspace, true);
    const cudaError_t e = launch_lmhead_verify(hidden, weight, d, logits, P, f[1], f[2], f[4], s);
    if (e == cudaErrorInvalidValue) return bad(SPECNG_EINVAL, "the tensor maps of hidden / weight could not be encoded");
    if (e != cudaSuccess) return fail_cuda(e, who);
    return SPECNG_OK;
}

int spec_verify_noalloc(const void* logits, int logits_dtype, int B, int K, int V, const int32_t* drafts,
                        const float* draft_probs, const int32_t* k, const int32_t* history, int64_t hist_stride,
                        const int32_t* lens, const specng_verify_params* params, int32_t* kv_len, float* ema,
                        int32_t* out_tokens, int32_t* out_accept_len, cudaStream_t s) {
    // every check comes before anything is enqueued on s
    VerifyDev P;
    bool f[5];
    int rc = verify_setup("spec_verify_noalloc", logits, logits_dtype, B, K, V, drafts, draft_probs, k, history,
                          hist_stride, lens, params, kv_len, ema, out_tokens, out_accept_len, s, &P, f);
    if (rc != SPECNG_OK) return rc;
    const size_t need = ws_layout(B, K, V).total;
    if (need > static_cast<size_t>(SPECNG_STATIC_SCRATCH_BYTES)) {
        std::snprintf(g_last_error, sizeof(g_last_error),
                      "spec_verify_noalloc: B=%d K=%d V=%d needs %zu bytes of scratch but the static scratch "
                      "holds %d; call spec_verify with a workspace instead", B, K, V, need,
                      SPECNG_STATIC_SCRATCH_BYTES);
        return SPECNG_ESMALL;
    }
    void* scratch = static_scratch_ptr();
    if (scratch == nullptr) return fail(SPECNG_ECUDA, "spec_verify_noalloc: scratch address lookup failed");
    const cudaError_t e = cudaMemsetAsync(scratch, 0, need, s);
    if (e != cudaSuccess) return fail_cuda(e, "spec_verify_noalloc");
    attach_workspace(P, scratch);
    return verify_launch(P, f, s, "spec_verify_noalloc");
}

int spec_append(int32_t* history, int64_t hist_stride, int32_t* lens, int64_t hist_cap, const int32_t* out_tokens,
                const int32_t* out_accept_len, int B, int K, cudaStream_t s) {
    if (history == nullptr || lens == nullptr || out_tokens == nullptr || out_accept_len == nullptr)
        return fail(SPECNG_EINVAL, "spec_append: NULL argument");
    if (B < 1 || K < 0 || K > SPECNG_MAX_K) return fail(SPECNG_EINVAL, "spec_append: B or K out of range");
    if (hist_stride < 1 || hist_cap < 0 || hist_cap > hist_stride)
        return fail(SPECNG_EINVAL, "spec_append: need 0 <= hist_cap <= hist_stride");
    const cudaError_t e = launch_spec_append(history, hist_stride, lens, hist_cap, out_tokens, out_accept_len, B, K,
                                             status_ptr(), s);
    if (e != cudaSuccess) return fail_cuda(e, "spec_append");
    return SPECNG_OK;
}

int spec_commit(specng_ngram* table, int32_t* history, int64_t hist_stride, int32_t* lens, int64_t hist_cap,
                const int32_t* out_tokens, const int32_t* out_accept_len, int B, int K, int max_k,
                const int32_t* k_limit, const int32_t* fallback, int32_t* out_drafts, int32_t* out_k,
                cudaStream_t s) {
    if (table == nullptr || history == nullptr || lens == nullptr || out_tokens == nullptr ||
        out_accept_len == nullptr || out_k == nullptr)
        return fail(SPECNG_EINVAL, "spec_commit: NULL argument");
    if (B != table->dev.B) return fail(SPECNG_EINVAL, "spec_commit: B differs from the table's B");
    if (K < 0 || K > SPECNG_MAX_K) return fail(SPECNG_EINVAL, "spec_commit: K outside [0, 16]");
    if (max_k < 0 || max_k > SPECNG_MAX_K) return fail(SPECNG_EINVAL, "spec_commit: max_k outside [0, 16]");
    if (max_k > 0 && out_drafts == nullptr) return fail(SPECNG_EINVAL, "spec_commit: out_drafts is NULL");
    if (hist_stride < 1 || hist_stride > SPECNG_NGRAM_MAX_POS)
        return fail(SPECNG_EINVAL, "spec_commit: hist_stride outside [1, 2^24]");
    if (hist_cap < 0 || hist_cap > hist_stride) return fail(SPECNG_EINVAL, "spec_commit: need 0 <= hist_cap <= hist_stride");
    const cudaError_t e = launch_spec_commit(table->dev, history, hist_stride, lens, hist_cap, out_tokens,
                                             out_accept_len, K, max_k, k_limit, fallback, out_drafts, out_k, s);
    if (e != cudaSuccess) return fail_cuda(e, "spec_commit");
    return SPECNG_OK;
}

int specng_get_counters(uint32_t* counts, int n, int clear) {
    if (counts == nullptr || n < 0 || n > SPECNG_DIAG_N) return fail(SPECNG_EINVAL, "specng_get_counters: bad argument");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda(e, "specng_get_counters");
    unsigned v[SPECNG_DIAG_N] = {};
    e = cudaMemcpyFromSymbol(v, g_diag_counters, sizeof(v));
    if (e != cudaSuccess) return fail_cuda(e, "specng_get_counters");
    for (int i = 0; i < n; ++i) counts[i] = v[i];
    if (clear) {
        const unsigned z[SPECNG_DIAG_N] = {};
        e = cudaMemcpyToSymbol(g_diag_counters, z, sizeof(z));
        if (e != cudaSuccess) return fail_cuda(e, "specng_get_counters");
    }
    return SPECNG_OK;
}

int specng_philox4x32_10(const uint32_t* ctr, uint64_t seed, uint32_t* out, int64_t n, cudaStream_t s) {
    if (ctr == nullptr || out == nullptr || n < 0) return fail(SPECNG_EINVAL, "specng_philox4x32_10: bad argument");
    if (!aligned16(ctr) || !aligned16(out)) return fail(SPECNG_EALIGN, "specng_philox4x32_10: 16-byte alignment");
    if (n == 0) return SPECNG_OK;
    const cudaError_t e = launch_philox(ctr, seed, out, n, s);
    if (e != cudaSuccess) return fail_cuda(e, "specng_philox4x32_10");
    return SPECNG_OK;
}

}  // extern "C"
