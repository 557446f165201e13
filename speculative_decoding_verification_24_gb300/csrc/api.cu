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

extern "C" sv_status spec_verify_ex(const sv_verify_args* a) {
    if (!a) return SV_ERR_NULL;
    if (!a->target_logits || !a->draft_tokens || !a->out_tokens || !a->out_n_accepted)
        return SV_ERR_NULL;
    if (a->B < 1 || a->K < 1 || a->K > 31 || a->V < 2) return SV_ERR_SHAPE;
    if (a->dtype != SV_F32 && a->dtype != SV_BF16) return SV_ERR_DTYPE;
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
    const size_t es = (size_t)esize_of(a->dtype);
    if (!aligned(a->target_logits, es) || (a->draft_logits && !aligned(a->draft_logits, es)) ||
        !aligned(a->draft_tokens, 4) || !aligned(a->out_tokens, 4) || !aligned(a->out_n_accepted, 4) ||
        (a->modes && !aligned(a->modes, 4)) || (a->seq_ids && !aligned(a->seq_ids, 8)) ||
        (a->out_p_target && !aligned(a->out_p_target, 4)) ||
        (a->out_p_draft && !aligned(a->out_p_draft, 4)) ||
        (a->out_residual_mass && !aligned(a->out_residual_mass, 4)) ||
        (a->status_word && !aligned(a->status_word, 4)))
        return SV_ERR_ALIGN;
    if (!valid_cluster_request(a->cluster_size)) return SV_ERR_CONFIG;
    // The grid holds B * cluster_size CTAs; keep it inside one dimension.
    if ((long long)a->B * 16 > 0x7FFFFFFFLL) return SV_ERR_SHAPE;

    int sms = 0;
    sv_status st = check_device(&sms);
    if (st != SV_OK) return st;

    const int cs_min = sv::min_cluster_size(a->V, (int)es);
    if (cs_min == 0) return SV_ERR_SHAPE;
    if (a->cluster_size && a->cluster_size < cs_min) return SV_ERR_CONFIG;
    int cs = a->cluster_size ? a->cluster_size
                             : sv::auto_cluster_size(a->B, a->V, (int)es, sms);
    const int usable = sv::usable_cluster_size((int)a->dtype, cs);
    if (usable == 0) return fail_cuda(cudaGetLastError());
    if (a->cluster_size && usable != cs) return SV_ERR_CONFIG;
    cs = usable;

    sv::VerifyParams p;
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
    p.status_word = a->status_word;
    cudaError_t e = sv::launch_verify_logits(p, (int)a->dtype, cs, (cudaStream_t)a->stream);
    if (e != cudaSuccess) return fail_cuda(e);
    return SV_OK;
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
    }
    return "unknown status";
}

extern "C" int sv_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" int sv_version(void) { return 100; }

extern "C" size_t sv_verify_args_size(void) { return sizeof(sv_verify_args); }

extern "C" size_t spec_verify_lmhead_workspace_bytes(int B, int K, int d, int V) {
    (void)B; (void)K; (void)d; (void)V;
    return 0;
}

extern "C" sv_status spec_verify_lmhead(const void* hidden, const void* W, const void* draft_logits,
                                        const int32_t* draft_tokens, int B, int K, int d, int V,
                                        sv_dtype draft_dtype, float temperature, sv_mode mode,
                                        uint64_t seed, void* workspace, size_t workspace_bytes,
                                        int32_t* out_tokens, int32_t* out_n_accepted,
                                        sv_stream_t stream) {
    (void)hidden; (void)W; (void)draft_logits; (void)draft_tokens; (void)B; (void)K; (void)d;
    (void)V; (void)draft_dtype; (void)temperature; (void)mode; (void)seed; (void)workspace;
    (void)workspace_bytes; (void)out_tokens; (void)out_n_accepted; (void)stream;
    return SV_ERR_NOT_IMPLEMENTED;
}
