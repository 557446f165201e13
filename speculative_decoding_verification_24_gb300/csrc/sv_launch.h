// Internal interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "specverify.h"

namespace sv {

// Arguments of the logits-path verify kernel, validated by the C-ABI layer.
struct VerifyParams {
    const void* target;        // [B, K+1, V]
    const void* draft;         // [B, K, V] or nullptr (greedy only)
    const int32_t* tokens;     // [B, K]
    const int32_t* modes;      // [B] or nullptr
    const uint64_t* seq_ids;   // [B] or nullptr
    int B, K, V;
    int mode;                  // used when modes == nullptr
    float c;                   // log2(e) / temperature
    uint64_t seed;
    int32_t* out_tokens;       // [B, K+1]
    int32_t* out_n_accepted;   // [B]
    float* out_p_target;       // [B, K] or nullptr
    float* out_p_draft;        // [B, K] or nullptr
    float* out_residual_mass;  // [B] or nullptr
    float* out_draw_edges;     // [B, 2] or nullptr: the draw target's distances to its interval's edges
    uint32_t* status_word;     // or nullptr
    int overlap_previous;      // inputs not written by the previous work on the stream
    const int32_t* draft_lens; // [B] per-sequence draft counts (0..K) or nullptr (all K)
    // Greedy tree verification when tree_parents != nullptr: K + 1 = N nodes,
    // tokens [B, N] (node tokens; node 0 the root), tree_parents [B, N].
    const int32_t* tree_parents;
    int32_t* out_last_node;    // [B] or nullptr (tree mode)
    int test_wait_timeout;     // tests of the failure path: a bounded wait that gives up
    int es_t, es_d;            // element sizes of the target and draft rows (debug build's checks)
    int test_debug_shrink;     // debug build's tests: the target's checked extent is halved
    // LM-head path: the target rows' statistics come as partials from the
    // GEMM epilogue, one per row and GEMM CTA (parts[cta * part_M + b * (K+1)
    // + i], part_tiles CTAs), written by the grid launched just before this
    // one on the stream; the target rows are then read only for the logits at
    // the draft tokens and the final draw, after that grid has completed.
    const float2* target_parts;
    int part_tiles, part_M;
    // With target_parts: the draft rows' partials too (parts[cta * B*K +
    // b * K + i]), or nullptr (the draft rows are streamed in pass 1).
    const float2* draft_parts;
};

// CTAs per cluster chosen from the shape when the caller asks for automatic.
int auto_cluster_size(int B, int V, int esize, int num_sms);

// Cluster size for a call that overlaps the previous one on its stream.
int overlap_cluster_size();

// Cluster size for the LM-head path's verify launch.
int fused_cluster_size(int B, int num_sms);

// Smallest cluster size whose per-CTA slice of a row fits the kernel's
// bookkeeping (0: the row is too long for any cluster size).
int min_cluster_size(int V, int esize);

// Whether the verify kernel is built for this (target, draft) pair of types:
// both fp32, both bf16, or fp32 target rows with bf16 draft rows.
bool supported_dtypes(int dtype_target, int dtype_draft);

// Largest cluster size <= cs that can be resident for these types (0 if none).
int usable_cluster_size(int dtype_target, int dtype_draft, int cs);

cudaError_t launch_verify_logits(const VerifyParams& p, int dtype_target, int dtype_draft, int cs,
                                 cudaStream_t stream);

// Grouped verify (plain calls): n_cl clusters of cs CTAs, cluster c taking
// the sequences the batch's snake order deals it. group_plan_fits: whether
// the kernel's tables hold such a plan for these sizes (can_sample: the call
// may have sample sequences); auto_group_plan: the plan a lone call uses by
// default, or false for one cluster per sequence.
bool group_plan_fits(int B, int K, bool can_sample, int V, int esize, int n_cl, int cs);
bool auto_group_plan(int B, int K, bool can_sample, int V, int esize, int num_sms, int& n_cl, int& cs);
cudaError_t launch_verify_grouped(const VerifyParams& p, int dtype_target, int dtype_draft, int n_cl, int cs,
                                  cudaStream_t stream);

// LM head: logits[M, V] (fp32) = hidden[M, d] . W[d, V] (bf16) on the tensor
// cores; 1 <= M <= 256, d a multiple of 64, V a multiple of 8, 16-byte
// aligned bases.
constexpr int PL_MAX_NGRAM = 16;
constexpr int PL_MAX_DRAFTS = 64;
cudaError_t launch_prompt_lookup(const int32_t* tokens, const int32_t* lengths, int B, int L_max,
                                 int max_ngram, int n_drafts, int32_t* out_drafts, int32_t* out_n,
                                 cudaStream_t stream);

cudaError_t launch_commit(int32_t* tokens, int32_t* lengths, int B, int L_max, const int32_t* out_tokens,
                          const int32_t* n_accepted, int K, int32_t* out_n_committed, cudaStream_t stream);

// With parts != nullptr the epilogue also reduces every row over each
// 128-column tile and merges the tiles of each CTA in tile order, writing one
// partial per row and CTA (parts[cta * M + m], *grid_out CTAs): base-2
// softmax partials (R, s) at scale c = log2(e) / T when part_soft, else
// (max, lowest index). With dp != nullptr (sample mode) two otherwise idle
// warps do the same for the draft rows (dparts[cta * Md + m]).
constexpr int LM_TILE_V = 128;
struct LmDraftParts {
    const void* draft;  // [Md, V], fp32 or bf16
    int Md, draft_f32;
    float2* dparts;     // [tiles, Md]
};
cudaError_t launch_lmhead_gemm(const void* hidden, const void* W, int M, int d, int V, float* out,
                               float2* parts, float c, int part_soft, const LmDraftParts* dp,
                               uint32_t* status, cudaStream_t stream, int* grid_out = nullptr);

}  // namespace sv
