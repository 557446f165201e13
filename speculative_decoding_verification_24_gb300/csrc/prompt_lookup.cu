// Prompt lookup drafting on the GPU ("Inference-4" (brunomaga.github.io),
// section "Prompt lookup decoding"): the drafts are the tokens that followed
// the most recent earlier occurrence of the sequence's last n-gram, trying
// n = max_ngram first; none when no n-gram of length 1..max_ngram recurs.
//
// One CTA per sequence. A window that ends at position e (e <= L-2, so it
// ends before the last token) matches the last n tokens for every n up to
// ml(e), the length of the common suffix of seq[..e] and seq[..L-1] (capped
// at max_ngram). The n that wins is the largest ml over all e, and its most
// recent window has the largest e among those: so one max-reduction of the
// key (ml(e), e) over all positions gives both. The drafts are then
// seq[e+1 .. e+n_drafts], cut at L.
#include <cstdint>

#include "sv_device.cuh"
#include "sv_launch.h"

namespace sv {

constexpr int PL_THREADS = 256;

__global__ void __launch_bounds__(PL_THREADS) prompt_lookup_kernel(const int32_t* tokens, const int32_t* lengths,
                                                                   int L_max, int max_ngram, int n_drafts,
                                                                   int32_t* out_drafts, int32_t* out_n) {
    __shared__ int32_t suffix[PL_MAX_NGRAM];
    __shared__ long long warp_best[PL_THREADS / 32];
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t* seq = tokens + (size_t)b * L_max;
    int32_t* out = out_drafts + (size_t)b * n_drafts;
    const int L = __ldg(lengths + b);
    const bool valid = L >= 0 && L <= L_max;
    if (valid && tid < max_ngram && tid < L) suffix[tid] = __ldg(seq + (L - 1 - tid));
    __syncthreads();
    if (!valid) {
        for (int i = tid; i < n_drafts; i += PL_THREADS) out[i] = -1;
        if (tid == 0) out_n[b] = -1;
        return;
    }
    long long best = -1;  // (ml << 32) | e, the largest over this thread's windows
    for (int e = tid; e <= L - 2; e += PL_THREADS) {
        int ml = 0;
        while (ml < max_ngram && e - ml >= 0 && __ldg(seq + (e - ml)) == suffix[ml]) ++ml;
        const long long key = ((long long)ml << 32) | (unsigned)e;
        best = key > best ? key : best;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const long long other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        best = other > best ? other : best;
    }
    if (lane == 0) warp_best[warp] = best;
    __syncthreads();
    if (warp == 0) {
        best = lane < PL_THREADS / 32 ? warp_best[lane] : -1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const long long other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
            best = other > best ? other : best;
        }
        const int ml = best < 0 ? 0 : (int)(best >> 32);
        const int e = best < 0 ? -1 : (int)(best & 0xFFFFFFFFLL);
        // drafts: seq[e+1 .. e+n_drafts], cut at the end of the sequence
        const int avail = ml > 0 ? min(n_drafts, L - 1 - e) : 0;
        for (int i = lane; i < n_drafts; i += 32) out[i] = i < avail ? __ldg(seq + (e + 1 + i)) : -1;
        if (lane == 0) out_n[b] = avail;
    }
}

cudaError_t launch_prompt_lookup(const int32_t* tokens, const int32_t* lengths, int B, int L_max,
                                 int max_ngram, int n_drafts, int32_t* out_drafts, int32_t* out_n,
                                 cudaStream_t stream) {
    prompt_lookup_kernel<<<B, PL_THREADS, 0, stream>>>(tokens, lengths, L_max, max_ngram, n_drafts,
                                                       out_drafts, out_n);
    return cudaGetLastError();
}

}  // namespace sv

namespace sv {

// Commit step of a decode loop: sequence b appends its n_accepted[b] accepted
// drafts and the token after them (out_tokens[b, 0..n]) to its context and
// advances its length, up to L_max. One warp per sequence (K + 1 <= 32).
__global__ void commit_kernel(int32_t* tokens, int32_t* lengths, int B, int L_max, const int32_t* out_tokens,
                              const int32_t* n_accepted, int K, int32_t* out_n_committed) {
    const int b = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (b >= B) return;
    const int n = __ldg(n_accepted + b);
    const int L = lengths[b];
    const bool ok = n >= 0 && n <= K && L >= 0 && L <= L_max;
    const int c = ok ? min(n + 1, L_max - L) : 0;
    if (lane < c) tokens[(size_t)b * L_max + L + lane] = __ldg(out_tokens + (size_t)b * (K + 1) + lane);
    __syncwarp();
    if (lane == 0) {
        if (ok) lengths[b] = L + c;
        if (out_n_committed) out_n_committed[b] = ok ? c : -1;
    }
}

cudaError_t launch_commit(int32_t* tokens, int32_t* lengths, int B, int L_max, const int32_t* out_tokens,
                          const int32_t* n_accepted, int K, int32_t* out_n_committed, cudaStream_t stream) {
    constexpr int WARPS = 8;
    commit_kernel<<<(B + WARPS - 1) / WARPS, WARPS * 32, 0, stream>>>(tokens, lengths, B, L_max, out_tokens,
                                                                     n_accepted, K, out_n_committed);
    return cudaGetLastError();
}

}  // namespace sv
