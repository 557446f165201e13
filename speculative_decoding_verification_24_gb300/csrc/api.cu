// C ABI of libspecverify: argument validation, device checks and dispatch.
// Every entry point validates on the host, returns before any launch on a
// host-detectable error, and otherwise enqueues its kernels on the caller's
// stream without synchronising.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "specverify.h"
#include "sv_launch.h"

namespace {

thread_local int g_last_cuda_error = 0;

constexpr int kMaxDevices = 64;
// Per device: 0 unknown, 1 supported, 2 unsupported; plus its SM count.
std::atomic<int> g_dev_state[kMaxDevices];
std::atomic<int> g_dev_sms[kMaxDevices];

sv_status fail_cuda(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return SV_ERR_CUDA;
}

// The current device must be compute capability 10.3 (the library is built
// for sm_103a only). Returns its SM count through *sms.
sv_status check_device(int* sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return SV_ERR_ARCH;
    int state = g_dev_state[dev].load(std::memory_order_acquire);
    if (state == 0) {
        int major = 0, minor = 0, n = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return fail_cuda(e);
        state = (major == 10 && minor == 3) ? 1 : 2;
        g_dev_sms[dev].store(n, std::memory_order_relaxed);
        g_dev_state[dev].store(state, std::memory_order_release);
    }
    if (state != 1) return SV_ERR_ARCH;
    *sms = g_dev_sms[dev].load(std::memory_order_relaxed);
    return SV_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int esize_of(sv_dtype d) { return d == SV_BF16 ? 2 : 4; }

bool valid_cluster_request(int cs) { return cs == 0 || cs == 1 || cs == 2 || cs == 4 || cs == 8 || cs == 16; }

}  // namespace

// The verify step over logits in device memory; the target rows have type
// dtype_t and the draft rows type dtype_d (equal, or fp32 target with bf16
// draft rows for the LM-head path).
// target_parts: the LM-head path's per-tile target-row partials (or NULL).
// plan_only: validate and choose the launch as a call would, report it there
// and enqueue nothing.
static sv_status verify_impl(const sv_verify_args* a, sv_dtype dtype_t, sv_dtype dtype_d,
                             const float2* target_parts = nullptr, int part_tiles = 0,
                             const float2* draft_parts = nullptr, sv_verify_plan* plan_only = nullptr) {
    if (!a) return SV_ERR_NULL;
    if (!a->target_logits || !a->draft_tokens || !a->out_tokens || !a->out_n_accepted)
        return SV_ERR_NULL;
    if (a->B < 1 || a->K < 1 || a->K > 31 || a->V < 2) return SV_ERR_SHAPE;
    if ((dtype_t != SV_F32 && dtype_t != SV_BF16) || (dtype_d != SV_F32 && dtype_d != SV_BF16) ||
        !sv::supported_dtypes(dtype_t, dtype_d))
        return SV_ERR_DTYPE;
    if (!a->modes && a->mode != SV_GREEDY && a->mode != SV_SAMPLE) return SV_ERR_MODE;
    if (!a->modes && a->mode == SV_SAMPLE && !a->draft_logits) return SV_ERR_NULL;
    const bool may_sample = a->modes != nullptr || a->mode == SV_SAMPLE;
    double c = 1.0;
    if (may_sample) {
        const double T = (double)a->temperature;
        if (!std::isfinite(T) || !(T > 0.0)) return SV_ERR_TEMPERATURE;
        c = 1.4426950408889634 / T;  // log2(e) / T
        if (!std::isfinite((float)c)) return SV_ERR_TEMPERATURE;
    }
    const size_t es_t = (size_t)esize_of(dtype_t), es_d = (size_t)esize_of(dtype_d);
    if (!aligned(a->target_logits, es_t) || (a->draft_logits && !aligned(a->draft_logits, es_d)) ||
        !aligned(a->draft_tokens, 4) || !aligned(a->out_tokens, 4) || !aligned(a->out_n_accepted, 4) ||
        (a->modes && !aligned(a->modes, 4)) || (a->seq_ids && !aligned(a->seq_ids, 8)) ||
        (a->draft_lens && !aligned(a->draft_lens, 4)) ||
        (a->out_p_target && !aligned(a->out_p_target, 4)) ||
        (a->out_p_draft && !aligned(a->out_p_draft, 4)) ||
        (a->out_residual_mass && !aligned(a->out_residual_mass, 4)) ||
        (a->out_draw_edges && !aligned(a->out_draw_edges, 4)) ||
        (a->status_word && !aligned(a->status_word, 4)))
        return SV_ERR_ALIGN;
    if (!valid_cluster_request(a->cluster_size)) return SV_ERR_CONFIG;
    // The grid holds B * cluster_size CTAs; keep it inside one dimension.
    if ((long long)a->B * 16 > 0x7FFFFFFFLL) return SV_ERR_SHAPE;

    int sms = 0;
    sv_status st = check_device(&sms);
    if (st != SV_OK) return st;

    const int cs_min = sv::min_cluster_size(a->V, (int)es_t);
    if (cs_min == 0) return SV_ERR_SHAPE;
    if (a->cluster_size && a->cluster_size < cs_min) return SV_ERR_CONFIG;
    int cs = a->cluster_size;
    if (!cs) {
        if (target_parts) {
            cs = sv::fused_cluster_size(a->B, sms);
        } else if (a->flags & SV_ARG_OVERLAP_PREVIOUS) {
            cs = sv::overlap_cluster_size();
        } else {
            cs = sv::auto_cluster_size(a->B, a->V, (int)es_t, sms);
        }
        if (cs < cs_min) cs = cs_min;
    }
    const int usable = sv::usable_cluster_size((int)dtype_t, (int)dtype_d, cs);
    if (usable == 0) return fail_cuda(cudaGetLastError());
    if (a->cluster_size && usable != cs) return SV_ERR_CONFIG;
    cs = usable;

    // Several sequences per cluster (plain calls): asked for, or automatic
    // when it spreads a large batch evenly over the SMs.
    const bool plain = !target_parts && !(a->flags & SV_ARG_OVERLAP_PREVIOUS);
    if (a->seqs_per_cluster < 0 || a->seqs_per_cluster > 8 || (a->seqs_per_cluster > 1 && !plain))
        return SV_ERR_CONFIG;
    int n_cl = 0, gcs = 0;
    bool grouped = false;
    if (plain && a->seqs_per_cluster > 1) {
        gcs = a->cluster_size ? a->cluster_size : 8;
        n_cl = (a->B + a->seqs_per_cluster - 1) / a->seqs_per_cluster;
        if (!sv::group_plan_fits(a->B, a->K, may_sample, a->V, (int)es_t, n_cl, gcs)) return SV_ERR_CONFIG;
        if (sv::usable_cluster_size((int)dtype_t, (int)dtype_d, gcs) != gcs) return SV_ERR_CONFIG;
        grouped = true;
    } else if (plain && a->seqs_per_cluster == 0 && a->cluster_size == 0) {
        grouped = sv::auto_group_plan(a->B, a->K, may_sample, a->V, (int)es_t, sms, n_cl, gcs) &&
                  sv::usable_cluster_size((int)dtype_t, (int)dtype_d, gcs) == gcs;
    }

    if (plan_only) {
        plan_only->grouped = grouped ? 1 : 0;
        plan_only->clusters = grouped ? n_cl : a->B;
        plan_only->cluster_size = grouped ? gcs : cs;
        plan_only->max_seqs_per_cluster = grouped ? (a->B + n_cl - 1) / n_cl : 1;
        return SV_OK;
    }

    sv::VerifyParams p = {};
    p.target = a->target_logits;
    p.draft = a->draft_logits;
    p.tokens = a->draft_tokens;
    p.modes = a->modes;
    p.seq_ids = a->seq_ids;
    p.B = a->B;
    p.K = a->K;
    p.V = a->V;
    p.mode = (int)a->mode;
    p.c = (float)c;
    p.seed = a->seed;
    p.out_tokens = a->out_tokens;
    p.out_n_accepted = a->out_n_accepted;
    p.out_p_target = a->out_p_target;
    p.out_p_draft = a->out_p_draft;
    p.out_residual_mass = a->out_residual_mass;
    p.out_draw_edges = a->out_draw_edges;
    p.status_word = a->status_word;
    p.overlap_previous = (a->flags & SV_ARG_OVERLAP_PREVIOUS) != 0;
    p.test_wait_timeout = (a->flags & SV_ARG_TEST_WAIT_TIMEOUT) != 0;
    p.test_debug_shrink = (a->flags & SV_ARG_TEST_DEBUG_SHRINK) != 0;
    p.es_t = (int)es_t;
    p.es_d = (int)es_d;
    p.draft_lens = a->draft_lens;
    p.target_parts = target_parts;
    p.part_tiles = part_tiles;
    p.part_M = a->B * (a->K + 1);
    p.draft_parts = draft_parts;
    cudaError_t e = grouped ? sv::launch_verify_grouped(p, (int)dtype_t, (int)dtype_d, n_cl, gcs, (cudaStream_t)a->stream)
                            : sv::launch_verify_logits(p, (int)dtype_t, (int)dtype_d, cs, (cudaStream_t)a->stream);
    if (e != cudaSuccess) return fail_cuda(e);
    return SV_OK;
}

extern "C" sv_status spec_verify_ex(const sv_verify_args* a) {
    if (!a) return SV_ERR_NULL;
    return verify_impl(a, a->dtype, a->dtype);
}

extern "C" sv_status spec_verify_plan(const sv_verify_args* a, sv_verify_plan* plan) {
    if (!a || !plan) return SV_ERR_NULL;
    return verify_impl(a, a->dtype, a->dtype, nullptr, 0, nullptr, plan);
}

extern "C" sv_status spec_verify(const void* target_logits, const void* draft_logits,
                                 const int32_t* draft_tokens, int B, int K, int V, sv_dtype dtype,
                                 float temperature, sv_mode mode, uint64_t seed, int32_t* out_tokens,
                                 int32_t* out_n_accepted, sv_stream_t stream) {
    sv_verify_args a = {};
    a.target_logits = target_logits;
    a.draft_logits = draft_logits;
    a.draft_tokens = draft_tokens;
    a.B = B;
    a.K = K;
    a.V = V;
    a.dtype = dtype;
    a.temperature = temperature;
    a.mode = mode;
    a.seed = seed;
    a.out_tokens = out_tokens;
    a.out_n_accepted = out_n_accepted;
    a.stream = stream;
    return spec_verify_ex(&a);
}

extern "C" const char* sv_status_string(sv_status s) {
    switch (s) {
        case SV_OK: return "ok";
        case SV_ERR_NULL: return "a required pointer is NULL";
        case SV_ERR_SHAPE: return "shape out of range";
        case SV_ERR_DTYPE: return "unknown dtype";
        case SV_ERR_TEMPERATURE: return "temperature must be finite and > 0 in sample mode";
        case SV_ERR_WORKSPACE: return "workspace missing or too small";
        case SV_ERR_ARCH: return "the current device is not compute capability 10.3 (sm_103a)";
        case SV_ERR_CUDA: return "CUDA runtime error (see sv_last_cuda_error)";
        case SV_ERR_MODE: return "unknown mode";
        case SV_ERR_ALIGN: return "pointer not aligned to its element size";
        case SV_ERR_CONFIG: return "requested launch configuration cannot be used";
        case SV_ERR_NOT_IMPLEMENTED: return "not implemented";
        case SV_ERR_SCRATCH_LIMIT:
            return "the LM-head workspace (logits and per-tile partials) exceeds the static scratch "
                   "(SV_LMHEAD_SCRATCH_BYTES)";
    }
    return "unknown status";
}

extern "C" int sv_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" int sv_version(void) { return 102; }

extern "C" size_t sv_verify_args_size(void) { return sizeof(sv_verify_args); }

extern "C" sv_status spec_verify_tree(const void* target_logits, sv_dtype dtype,
                                      const int32_t* tree_tokens, const int32_t* tree_parents, int B,
                                      int N, int V, int32_t* out_tokens, int32_t* out_n_accepted,
                                      int32_t* out_last_node, sv_stream_t stream) {
    if (!target_logits || !tree_tokens || !tree_parents || !out_tokens || !out_n_accepted) return SV_ERR_NULL;
    if (B < 1 || N < 1 || N > 32 || V < 2) return SV_ERR_SHAPE;
    if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
    if ((long long)B * 16 > 0x7FFFFFFFLL) return SV_ERR_SHAPE;
    const size_t es = (size_t)esize_of(dtype);
    if (!aligned(target_logits, es) || !aligned(tree_tokens, 4) || !aligned(tree_parents, 4) ||
        !aligned(out_tokens, 4) || !aligned(out_n_accepted, 4) || (out_last_node && !aligned(out_last_node, 4)))
        return SV_ERR_ALIGN;
    int sms = 0;
    sv_status st = check_device(&sms);
    if (st != SV_OK) return st;
    const int cs_min = sv::min_cluster_size(V, (int)es);
    if (cs_min == 0) return SV_ERR_SHAPE;
    const int cs = sv::usable_cluster_size((int)dtype, (int)dtype, sv::auto_cluster_size(B, V, (int)es, sms));
    if (cs == 0) return fail_cuda(cudaGetLastError());
    sv::VerifyParams p = {};
    p.target = target_logits;
    p.draft = nullptr;
    p.tokens = tree_tokens;
    p.B = B;
    p.K = N - 1;
    p.V = V;
    p.mode = SV_GREEDY;
    p.c = 1.0f;
    p.out_tokens = out_tokens;
    p.out_n_accepted = out_n_accepted;
    p.tree_parents = tree_parents;
    p.out_last_node = out_last_node;
    p.es_t = p.es_d = esize_of(dtype);
    cudaError_t e = sv::launch_verify_logits(p, (int)dtype, (int)dtype, cs, (cudaStream_t)stream);
    if (e != cudaSuccess) return fail_cuda(e);
    return SV_OK;
}

extern "C" sv_status spec_prompt_lookup(const int32_t* tokens, const int32_t* lengths, int B, int L_max,
                                        int max_ngram, int n_drafts, int32_t* out_drafts,
                                        int32_t* out_n_drafts, sv_stream_t stream) {
    if (!tokens || !lengths || !out_drafts || !out_n_drafts) return SV_ERR_NULL;
    if (B < 1 || L_max < 1 || max_ngram < 1 || max_ngram > sv::PL_MAX_NGRAM || n_drafts < 1 ||
        n_drafts > sv::PL_MAX_DRAFTS || B > 0x7FFFFFFF / 8)
        return SV_ERR_SHAPE;
    if (!aligned(tokens, 4) || !aligned(lengths, 4) || !aligned(out_drafts, 4) || !aligned(out_n_drafts, 4))
        return SV_ERR_ALIGN;
    int sms = 0;
    sv_status st = check_device(&sms);
    if (st != SV_OK) return st;
    cudaError_t e = sv::launch_prompt_lookup(tokens, lengths, B, L_max, max_ngram, n_drafts, out_drafts,
                                             out_n_drafts, (cudaStream_t)stream);
    if (e != cudaSuccess) return fail_cuda(e);
    return SV_OK;
}

extern "C" sv_status spec_commit(int32_t* tokens, int32_t* lengths, int B, int L_max,
                                 const int32_t* out_tokens, const int32_t* n_accepted, int K,
                                 int32_t* out_n_committed, sv_stream_t stream) {
    if (!tokens || !lengths || !out_tokens || !n_accepted) return SV_ERR_NULL;
    if (B < 1 || L_max < 1 || K < 0 || K > 31) return SV_ERR_SHAPE;
    if (!aligned(tokens, 4) || !aligned(lengths, 4) || !aligned(out_tokens, 4) || !aligned(n_accepted, 4) ||
        (out_n_committed && !aligned(out_n_committed, 4)))
        return SV_ERR_ALIGN;
    int sms = 0;
    sv_status st = check_device(&sms);
    if (st != SV_OK) return st;
    cudaError_t e = sv::launch_commit(tokens, lengths, B, L_max, out_tokens, n_accepted, K, out_n_committed,
                                      (cudaStream_t)stream);
    if (e != cudaSuccess) return fail_cuda(e);
    return SV_OK;
}

static size_t lmhead_logits_bytes(long long M, long long V) {
    return (size_t)(((M * V * 4) + 255) / 256 * 256);
}

// The LM-head verify's workspace: the fp32 logits [M, V], then room for one
// 8-byte partial per row and 128-column tile ([tiles, M]; the GEMM, one CTA
// per SM over at most that many tiles, uses the first rows), each part
// 256-aligned.
static long long lmhead_tiles(long long V) { return (V + sv::LM_TILE_V - 1) / sv::LM_TILE_V; }
static size_t lmhead_parts_bytes(long long M, long long V) {
    return (size_t)((lmhead_tiles(V) * M * 8 + 255) / 256 * 256);
}
// Then (sample mode) the draft rows' partials [tiles, B*K].
static size_t lmhead_workspace_bytes(long long B, long long K, long long V) {
    return lmhead_logits_bytes(B * (K + 1), V) + lmhead_parts_bytes(B * (K + 1), V) + lmhead_parts_bytes(B * K, V);
}

static sv_status check_lmhead_shape(const void* hidden, const void* W, long long M, int d, int V) {
    if (!hidden || !W) return SV_ERR_NULL;
    if (M < 1 || M > 256 || d < 64 || d % 64 != 0 || V < 8 || V % 8 != 0) return SV_ERR_SHAPE;
    if (!aligned(hidden, 16) || !aligned(W, 16)) return SV_ERR_ALIGN;
    return SV_OK;
}

extern "C" sv_status spec_lmhead_logits(const void* hidden, const void* W, int M, int d, int V,
                                        float* out, sv_stream_t stream) {
    sv_status st = check_lmhead_shape(hidden, W, M, d, V);
    if (st != SV_OK) return st;
    if (!out) return SV_ERR_NULL;
    if (!aligned(out, 4)) return SV_ERR_ALIGN;
    int sms = 0;
    if ((st = check_device(&sms)) != SV_OK) return st;
    cudaError_t e = sv::launch_lmhead_gemm(hidden, W, M, d, V, out, nullptr, 0.0f, 0, nullptr, nullptr,
                                           (cudaStream_t)stream);
    if (e != cudaSuccess) return fail_cuda(e);
    return SV_OK;
}

extern "C" size_t spec_verify_lmhead_workspace_bytes(int B, int K, int d, int V) {
    (void)d;
    if (B < 1 || K < 1 || V < 1) return 0;
    return lmhead_workspace_bytes(B, K, V);
}

extern "C" sv_status spec_verify_lmhead(const void* hidden, const void* W, const void* draft_logits,
                                        const int32_t* draft_tokens, int B, int K, int d, int V,
                                        sv_dtype draft_dtype, float temperature, sv_mode mode,
                                        uint64_t seed, void* workspace, size_t workspace_bytes,
                                        int32_t* out_tokens, int32_t* out_n_accepted,
                                        sv_stream_t stream) {
    if (B < 1 || K < 1 || K > 31) return SV_ERR_SHAPE;
    const long long M = (long long)B * (K + 1);
    sv_status st = check_lmhead_shape(hidden, W, M, d, V);
    if (st != SV_OK) return st;
    if (draft_dtype != SV_F32 && draft_dtype != SV_BF16) return SV_ERR_DTYPE;
    if (!workspace) return SV_ERR_WORKSPACE;
    if (workspace_bytes < lmhead_workspace_bytes(B, K, V)) return SV_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return SV_ERR_ALIGN;
    // validate the verify half before anything is launched
    sv_verify_args a = {};
    a.target_logits = workspace;
    a.draft_logits = draft_logits;
    a.draft_tokens = draft_tokens;
    a.B = B;
    a.K = K;
    a.V = V;
    a.dtype = SV_F32;
    a.temperature = temperature;
    a.mode = mode;
    a.seed = seed;
    a.out_tokens = out_tokens;
    a.out_n_accepted = out_n_accepted;
    a.stream = stream;
    if (!draft_tokens || !out_tokens || !out_n_accepted) return SV_ERR_NULL;
    if (mode != SV_GREEDY && mode != SV_SAMPLE) return SV_ERR_MODE;
    if (mode == SV_SAMPLE) {
        if (!draft_logits) return SV_ERR_NULL;
        if (!std::isfinite(temperature) || !(temperature > 0.0f)) return SV_ERR_TEMPERATURE;
    }
    int sms = 0;
    if ((st = check_device(&sms)) != SV_OK) return st;
    // the same scale as the verify kernel's: log2(e) / T, rounded once to float
    const float c = mode == SV_SAMPLE ? (float)(1.4426950408889634 / (double)temperature) : 0.0f;
    if (mode == SV_SAMPLE && !std::isfinite(c)) return SV_ERR_TEMPERATURE;
    char* ws = static_cast<char*>(workspace);
    float2* parts = reinterpret_cast<float2*>(ws + lmhead_logits_bytes(M, V));
    float2* dparts = reinterpret_cast<float2*>(ws + lmhead_logits_bytes(M, V) + lmhead_parts_bytes(M, V));
    sv::LmDraftParts dp{draft_logits, B * K, draft_dtype == SV_F32 ? 1 : 0, dparts};
    const bool sample = mode == SV_SAMPLE;
    int gemm_ctas = 0;
    // Greedy decisions and the token after them come from the (max, lowest
    // index) partials alone; only a sample call's final draw reads logits
    // (row j's), so a greedy call stores none of them.
    cudaError_t e = sv::launch_lmhead_gemm(hidden, W, (int)M, d, V, sample ? static_cast<float*>(workspace) : nullptr,
                                           parts, c,
                                           sample ? 1 : 0, sample ? &dp : nullptr, nullptr, (cudaStream_t)stream,
                                           &gemm_ctas);
    if (e != cudaSuccess) return fail_cuda(e);
    // the verify grid may start as the GEMM's CTAs finish; it waits for the
    // GEMM before it reads the logits and the partials (one per row and CTA)
    return verify_impl(&a, SV_F32, sample ? draft_dtype : SV_F32, parts, gemm_ctas, sample ? dparts : nullptr);
}

// ---------------------------------------------------------------------------
// LM-head verify with no allocation at all.
//
// Callers that cannot allocate device memory at verify time (a C host runtime
// without an allocator of its own; a serving loop that avoids cudaMalloc and
// cudaFree between steps because either may synchronise the whole device)
// get the fp32 target logits written to this fixed array instead of a
// workspace. It lives in this translation unit's device image, one copy per
// device, loaded with it; no call below allocates anything.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_lmhead_scratch[SV_LMHEAD_SCRATCH_BYTES];

static std::atomic<void*> g_scratch_addr[kMaxDevices];

// The scratch's device address on the current device, looked up once per
// device (with that device current) and cached. The first lookup on a device
// checks its compute capability first, so that a device this library was not
// built for reports SV_ERR_ARCH instead of failing to load the image.
static sv_status scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return SV_ERR_ARCH;
    void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        int sms = 0;
        const sv_status st = check_device(&sms);
        if (st != SV_OK) return st;
        e = cudaGetSymbolAddress(&p, g_lmhead_scratch);
        if (e != cudaSuccess) return fail_cuda(e);
        if (!p) return fail_cuda(cudaErrorInvalidSymbol);
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return SV_OK;
}

extern "C" sv_status spec_verify_lmhead_noalloc(const void* hidden, const void* W,
                                                const void* draft_logits, const int32_t* draft_tokens,
                                                int B, int K, int d, int V, sv_dtype draft_dtype,
                                                float temperature, sv_mode mode, uint64_t seed,
                                                int32_t* out_tokens, int32_t* out_n_accepted,
                                                sv_stream_t stream) {
    if (B < 1 || K < 1 || K > 31 || V < 1) return SV_ERR_SHAPE;
    // B*(K+1) <= 256 is checked by the callee; bound the product here first
    if ((long long)B * (K + 1) > 256) return SV_ERR_SHAPE;
    if (lmhead_workspace_bytes(B, K, V) > (size_t)SV_LMHEAD_SCRATCH_BYTES)
        return SV_ERR_SCRATCH_LIMIT;
    // every other argument is validated by spec_verify_lmhead before launching;
    // validate the cheap host-side ones first so that a bad call never loads
    // the device image
    sv_status st = check_lmhead_shape(hidden, W, (long long)B * (K + 1), d, V);
    if (st != SV_OK) return st;
    if (!draft_tokens || !out_tokens || !out_n_accepted) return SV_ERR_NULL;
    void* scratch = nullptr;
    if ((st = scratch_address(&scratch)) != SV_OK) return st;
    return spec_verify_lmhead(hidden, W, draft_logits, draft_tokens, B, K, d, V, draft_dtype,
                              temperature, mode, seed, scratch, (size_t)SV_LMHEAD_SCRATCH_BYTES,
                              out_tokens, out_n_accepted, stream);
}
