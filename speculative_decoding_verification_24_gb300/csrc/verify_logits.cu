// Verify kernel over logits in HBM: one thread-block cluster per sequence.
//
// What it computes follows "Inference-4" (brunomaga.github.io), section
// "Draft-model speculative decoding", and "Speculative decoding"
// (leoniemonigatti.com blog), section "Rejection sampling":
//   greedy  - accept drafts while x_i equals the argmax of target row i; emit
//             the argmax of the first mismatching row (or of row K);
//   sample  - accept x_i iff u_i * P_d,i(x_i) < P_t,i(x_i); at the first
//             rejection j draw from norm(max(0, P_t,j - P_d,j)); if all K pass
//             draw the bonus from P_t,K. Draws are inverse CDFs in index order.
//
// Layout of the work (one launch, no global scratch):
//   pass 1  Each of the CS CTAs of a cluster owns a contiguous slice of V and
//           streams that slice of every row the sequence needs (K+1 target
//           rows; plus K draft rows in sample mode). The slices' 16-byte
//           slots form one schedule cut into 4 KB chunks, row after row (a
//           row's last chunk may be shorter). Each of the 8 warps owns three
//           shared-memory stages and streams its own chunks: every 8th one,
//           or a contiguous run when the slices are short (see
//           stream_pass1). Bulk copies (cp.async.bulk, evict-first in L2, no
//           multicast) complete on the stage's mbarrier; the warp copies the
//           chunk into registers, refills the stage with its chunk three
//           ahead, then reduces: (R, s) base-2 softmax partials with packed
//           fp32x2 arithmetic for sample rows, (max, lowest index) for
//           greedy rows. Partial 16-byte slots at a row's two ends use plain
//           loads.
//   decide  Every CTA pushes its per-row partials into every CTA of the
//           cluster (distributed shared memory); after one cluster barrier
//           each CTA merges them in rank order (so all hold bit-identical
//           statistics), gathers the logits at the draft tokens, draws its
//           Philox uniforms and finds the first rejection with a warp ballot.
//           CTA 0 writes the outputs.
//   pass 2  Sample mode only: row j (target, and draft after a rejection)
//           streams through the same stages in 128-slot chunks; a warp sums
//           each chunk's draw mass in a fixed order (a warp scan per 32
//           slots). CTA totals are pushed cluster-wide; the CTA holding
//           u2 * total walks its chunk totals with a warp scan and one warp
//           re-reads that chunk to find the token.
//   Every mbarrier wait is bounded; a wait that gives up marks the sequence
//   invalid (SV_FLAG_TIMEOUT), and every warp waits for its own copies
//   before the CTA exits.
#include "verify_common.cuh"

#include <atomic>

namespace sv {

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
struct SeqShared {
    uint64_t full[NSTAGE];
    RowInfo rows[MAX_ROWS];
    float2 warp_part[NCW][MAX_ROWS];
    float2 edge_part[MAX_ROWS];
    float2 gathered[MAX_CS][MAX_ROWS];  // every CTA's partials, pushed by their owners
    float2 merged[MAX_ROWS];
    float p2_part[MAX_P2_CHUNKS];
    float p2_edge[2];
    unsigned char p2_seq0[NCW];         // each warp's fill count mod NBUF when pass 2 began
    float lt_x[MAX_K], ld_x[MAX_K];     // the logits at the draft tokens (captured in pass 1)
    float2 gathered_tot[2][MAX_CS];     // every CTA's draw mass (float-float), pushed by their owners
    float u_pos[MAX_K + 1], u2_pos[MAX_K + 1];  // Philox uniforms of positions 0..K
    // decision (identical in every CTA of the cluster)
    int j, valid, sample, use_d, err;
    float u2;
    SoftPart st, sd;
    ff total, tc;
    int cstar;
    int total_chunks;
    int seq_b;                          // the sequence this cluster verifies
    uint64_t never;                     // a barrier nothing completes (failure-path tests)
    // the final search in the CTA holding the draw
    int found, step_lp[P2_SLOTS / 32], step_hit[P2_SLOTS / 32];
    float step_tot[P2_SLOTS / 32];
    ff tw;
};

// Two CTAs per SM: 2 x (ring + this + 1 KB reserved) within 228 KB.
static_assert(2 * (RING_BYTES + sizeof(SeqShared) + 1024) <= 228 * 1024,
              "shared state too large for two CTAs per SM");

// Greedy tree verification ("Inference-4", section "Medusa": every candidate
// of the tree is verified in one pass and the longest accepted path is kept).
// Lane i holds node i (N <= 32): its token x_reg and parent; a node is
// accepted when its parent is and its token is the argmax of its parent's
// row. Acceptance and depth follow parent links, one level per step. The
// kept path ends at the deepest accepted node (lowest index among equally
// deep ones); the output is its tokens and the argmax of its own row.
__device__ __forceinline__ void tree_decide(const VerifyParams& p, SeqShared& sh, int b, int N, int V,
                                            int lane, int rank, bool mode_ok, int x_reg) {
    const bool node = lane < N && N <= 32;
    const int par = (lane > 0 && node) ? ld_in(p, p.tree_parents + (size_t)b * N + lane, -1) : -1;
    bool bad_row = false;
    if (node) {
        const ArgPart ap = as_arg(sh.merged[lane]);
        bad_row = !isfinite(ap.v) || ap.i < 0 || ap.i >= V;
    }
    const bool bad_link = lane > 0 && node && (par < 0 || par >= lane);
    const bool any_bad_row = __any_sync(FULL, bad_row), any_bad_link = __any_sync(FULL, bad_link);
    const int src = (par < 0 || bad_link) ? 0 : par;
    const int am_par = (lane > 0 && node && !bad_link) ? as_arg(sh.merged[src]).i : -1;
    const bool match = node && (lane == 0 || x_reg == am_par);
    bool acc = match;
    int depth = 0;
    for (int it = 1; it < N; ++it) {  // no path is longer than N - 1 links
        const bool acc_par = __shfl_sync(FULL, acc, src);
        const int d_par = __shfl_sync(FULL, depth, src);
        if (lane > 0 && node) {
            acc = match && acc_par;
            depth = d_par + 1;
        }
    }
    const bool acc_src = __shfl_sync(FULL, acc, src);  // every lane takes part in the shuffle
    const bool tested = lane > 0 && node && acc_src;
    const bool any_bad_token = __any_sync(FULL, tested && (x_reg < 0 || x_reg >= V));
    const bool invalid = !mode_ok || any_bad_row || any_bad_link || any_bad_token;
    int key = (acc && node) ? (depth << 6) | (63 - lane) : -1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) key = max(key, __shfl_xor_sync(FULL, key, o));
    const int last = invalid ? -1 : 63 - (key & 63);
    const int n = invalid ? -1 : key >> 6;
    // last < N and n < N by construction (key comes from a node lane); the
    // guards below keep every store inside the sequence's N outputs regardless
    if (lane == 0) {
        sh.sample = 0;
        sh.valid = !invalid;
    }
    if (rank != 0) return;
    if (p.overlap_previous) grid_dependency_wait();  // the stores below follow the previous call's
    int32_t* out = p.out_tokens + (size_t)b * N;
    if (!invalid) {
        int cur = last;
        for (int k = min(n, N) - 1; k >= 0; --k) {  // the path, from its last node up to the root
            const int tok = __shfl_sync(FULL, x_reg, cur & 31);
            const int up = __shfl_sync(FULL, par, cur & 31);
            if (lane == 0) st_out(p, out + k, tok);
            cur = up < 0 ? 0 : up;
        }
    }
    if (node && (invalid || lane >= n))
        st_out(p, out + lane, (!invalid && lane == n && last >= 0 && last < N) ? as_arg(sh.merged[last]).i : -1);
    if (lane == 0) {
        st_out(p, p.out_n_accepted + (b), n);
        if (p.out_last_node) st_out(p, p.out_last_node + (b), last);
        if (p.status_word && invalid)
            atomicOr(p.status_word, any_bad_link    ? (unsigned)SV_FLAG_BAD_TREE
                                    : any_bad_token ? (unsigned)SV_FLAG_BAD_TOKEN
                                                    : (unsigned)SV_FLAG_BAD_ROW);
        if (p.status_word && sh.err) atomicOr(p.status_word, (unsigned)SV_FLAG_TIMEOUT);
    }
}


// Where the draft token of row r lies in this CTA's pass-1 chunks: the chunk
// (or -1 when the token is not in the row's interior slots here), the byte
// offset of its element in the stage, and the token's position i. Row r is
// target row r (r < K) or draft row r - K - 1; row K has no draft token.
// x_reg: lane i holds draft token x_i. Called by the whole warp.
struct TokenSpot {
    int chunk, byte, i;
};

template <typename T>
__device__ __forceinline__ TokenSpot token_spot(const RowInfo& ri, int r, int K, int x_reg, int c0) {
    constexpr int E = Elem<T>::E;
    TokenSpot ts{-1, 0, -1};
    if (r == K) return ts;
    ts.i = r < K ? r : r - K - 1;
    const int x = __shfl_sync(FULL, x_reg, ts.i);
    if (x < 0) return ts;  // an invalid token (caught in the decision)
    const int slot = (x + ri.head) / E;
    if (slot < ri.ia || slot >= ri.ib) return ts;
    ts.chunk = c0 + (slot - ri.ia) / STAGE_SLOTS;
    ts.byte = ((slot - ri.ia) % STAGE_SLOTS) * 16 + ((x + ri.head) % E) * (int)sizeof(T);
    return ts;
}

// Lane 0 writes the logit at ts into every CTA of the cluster (exactly one
// CTA's slice holds any given element, so each value has one writer).
template <typename T>
__device__ __forceinline__ void capture_logit(SeqShared& sh, cg::cluster_group& cluster, int CS,
                                              const char* stage, const TokenSpot& ts, int K, int r) {
    const char* at = stage + ts.byte;
    float v;
    if constexpr (sizeof(T) == 4) v = *reinterpret_cast<const float*>(at);
    else v = __uint_as_float((uint32_t)(*reinterpret_cast<const unsigned short*>(at)) << 16);
    float* dst = r < K ? sh.lt_x : sh.ld_x;
    for (int cr = 0; cr < CS; ++cr) cluster.map_shared_rank(dst, cr)[ts.i] = v;
}

// As capture_logit for the partial edge slots: each lane holds one slot q
// (q < 0: none).
template <typename T>
__device__ __forceinline__ void capture_edge_logit(SeqShared& sh, cg::cluster_group& cluster, int CS,
                                                   const uint4& d, int q, int r, int K, int x_reg,
                                                   int head, int lane) {
    constexpr int E = Elem<T>::E;
    if (r == K) return;
    const int i = r < K ? r : r - K - 1;
    const int x = __shfl_sync(FULL, x_reg, i);
    if (x < 0 || q < 0 || (x + head) / E != q) return;
    const float v = elem_rt<T>(d, (x + head) % E);
    float* dst = r < K ? sh.lt_x : sh.ld_x;
    for (int cr = 0; cr < CS; ++cr) cluster.map_shared_rank(dst, cr)[i] = v;
}

// Pass 1 of one warp: chunks warp, warp + NCW, ... of the schedule, buffered
// in the warp's NBUF stages. Writes one partial per row it saw.
constexpr int RUN_ROW_CHUNKS = 64;  // row slices shorter than this on average: contiguous runs

template <typename TT, typename TD, bool SAMPLE, typename WhileWaiting>
__device__ __forceinline__ void stream_pass1(const VerifyParams& p, SeqShared& sh, WarpRing& wr, char* ring, int nchunks,
                                             int nrows, float c, int warp, int lane, uint32_t& seq,
                                             cg::cluster_group& cluster, int CS, int K, int x_reg,
                                             WhileWaiting&& while_waiting) {
    // The warp's chunks: every NCW-th chunk (the CTA's warps read neighbouring
    // chunks, and when all chunks fit the ring at once, chunk c lands in stage
    // c, where the second pass may read row j back), unless the CTA's slices of
    // the rows are short: then a warp would change rows (a butterfly flush of
    // its partial each time) every few chunks, and it takes a contiguous run
    // instead. Measured on GB300 with runs for slices under RUN_ROW_CHUNKS
    // chunks, against every NCW-th chunk: back to back B=8 x 11 rows of 32000
    // fp32 1.91 -> 1.77 us, B=64 x (5 or 9) rows of 128256 bf16 19.6 -> 18.9
    // us, trees of 32 rows on clusters of 4 85.8 -> 82.0 us; with runs for
    // every size, 17 rows of 151936 bf16 (75 chunks a row) went 192.4 ->
    // 193.3 us.
    int first = warp, end = nchunks, step = NCW;
    if (nchunks > NSTAGE && nchunks < RUN_ROW_CHUNKS * nrows) {
        split_range(nchunks, warp, NCW, first, end);
        step = 1;
    }
    FillCursor fill_rc{{-1, 0, 0}, nullptr, 0, 0};
    RowCursor rc{-1, 0, 0};
    for (int j = 0; j < NBUF; ++j) {
        const int chunk = first + step * j;
        if (chunk < end) fill_pass1(p, sh, wr, ring, seq + j, chunk, fill_rc, lane);
    }
    while_waiting();  // work that fits in the first copies' latency
    int cur_row = -1, ia = 0, ib = 0, head = 0;
    TokenSpot ts{-1, 0, -1};
    SoftAcc sa = soft_acc_empty();
    ArgAcc aa = arg_acc_empty();
    for (int chunk = first; chunk < end; chunk += step, ++seq) {
        seek_row(rc, sh.rows, chunk);
        if (rc.r != cur_row) {  // a new row: flush the last one, look the new one up once
            if (cur_row >= 0) {
                if (std::is_same<TT, TD>::value || cur_row <= K) flush_row<TT, SAMPLE>(sh, warp, lane, cur_row, sa, aa, head);
                else flush_row<TD, SAMPLE>(sh, warp, lane, cur_row, sa, aa, head);
            }
            sa = soft_acc_empty();
            aa = arg_acc_empty();
            cur_row = rc.r;
            const RowInfo ri = sh.rows[cur_row];
            ia = ri.ia;
            ib = ri.ib;
            head = ri.head;
            if (SAMPLE)
                ts = (std::is_same<TT, TD>::value || cur_row <= K) ? token_spot<TT>(ri, cur_row, K, x_reg, rc.c0)
                                                                  : token_spot<TD>(ri, cur_row, K, x_reg, rc.c0);
        }
        if (!wr.wait(sh, seq)) {
            atomicExch(&sh.err, 1);
            break;
        }
        const int q0 = ia + (chunk - rc.c0) * STAGE_SLOTS;
        const int n = min(STAGE_SLOTS, ib - q0);
        const char* stage = wr.stage(ring, seq);
        uint4 d[CHUNK_LANE_SLOTS];
        if (n == STAGE_SLOTS) {  // a full chunk (warp-uniform): no per-slot select
#pragma unroll
            for (int u = 0; u < CHUNK_LANE_SLOTS; ++u) d[u] = lds128(stage + (u * 32 + lane) * 16);
        } else {  // slots past the chunk's end read as -inf of the row's own type
            const uint4 pad = (std::is_same<TT, TD>::value || cur_row <= K) ? neg_inf_slot<TT>() : neg_inf_slot<TD>();
#pragma unroll
            for (int u = 0; u < CHUNK_LANE_SLOTS; ++u) {
                const int i = u * 32 + lane;
                d[u] = i < n ? lds128(stage + i * 16) : pad;
            }
        }
        if (SAMPLE && chunk == ts.chunk && lane == 0) {
            if (std::is_same<TT, TD>::value || cur_row <= K) capture_logit<TT>(sh, cluster, CS, stage, ts, K, cur_row);
            else capture_logit<TD>(sh, cluster, CS, stage, ts, K, cur_row);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (chunk + NBUF * step < end)
            fill_pass1(p, sh, wr, ring, seq + NBUF, chunk + NBUF * step, fill_rc, lane);
        if (std::is_same<TT, TD>::value || cur_row <= K) reduce_chunk<TT, SAMPLE>(sa, aa, d, n, q0, c, lane);
        else reduce_chunk<TD, SAMPLE>(sa, aa, d, n, q0, c, lane);
    }
    if (cur_row >= 0) {
        if (std::is_same<TT, TD>::value || cur_row <= K) flush_row<TT, SAMPLE>(sh, warp, lane, cur_row, sa, aa, head);
        else flush_row<TD, SAMPLE>(sh, warp, lane, cur_row, sa, aa, head);
    }
}

// One partial edge slot per lane (lane 0: the low end, lane 1: the high end of
// this CTA's slice of row r), reduced like the chunks.
template <typename T, bool SAMPLE>
__device__ __forceinline__ float2 edge_row(const VerifyParams& p, SeqShared& sh, const T* row, const RowInfo& ri, int r,
                                           int K, int V, float c, int lane, cg::cluster_group& cluster,
                                           int CS, int x_reg) {
    const RowGeom g{ri.base, ri.head, 0};
    uint4 d[1];
    int qs[1];
    qs[0] = lane == 0 ? ri.edge_lo : lane == 1 ? ri.edge_hi : -1;
    d[0] = qs[0] >= 0 ? load_slot<T>(p, g, row, V, qs[0]) : neg_inf_slot<T>();
    if (SAMPLE) {
        capture_edge_logit<T>(sh, cluster, CS, d[0], qs[0], r, K, x_reg, ri.head, lane);
        SoftAcc ea = soft_acc_empty();
        soft_group<T, 1>(ea, d, c);
        SoftPart pp{ea.R, soft_acc_sum(ea)};
        if (ea.R == -INFINITY) pp.s = 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            pp = merge_soft(pp, SoftPart{__shfl_xor_sync(FULL, pp.R, o), __shfl_xor_sync(FULL, pp.s, o)});
        return pack(pp);
    } else {
        ArgPart ea{-INFINITY, INT_MAX};
        arg_group<T, 1>(ea, d, qs, ri.head);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            ea = merge_arg(ea, ArgPart{__shfl_xor_sync(FULL, ea.v, o), __shfl_xor_sync(FULL, ea.i, o)});
        return pack(ea);
    }
}

// Partial slots at the two ends of this CTA's slices (warp 0).
template <typename TT, typename TD, bool SAMPLE>
__device__ __forceinline__ void edge_pass1(const VerifyParams& p, SeqShared& sh, const TT* tgt, const TD* drf, int b, int K,
                                           int Kb, int V, int nrows, float c, int lane,
                                           cg::cluster_group& cluster, int CS, int x_reg) {
    for (int r = 0; r < nrows; ++r) {
        const RowInfo ri = sh.rows[r];
        float2 part;
        if (ri.edge_lo < 0 && ri.edge_hi < 0) {
            part = SAMPLE ? pack(SoftPart{-INFINITY, 0.0f}) : pack(ArgPart{-INFINITY, INT_MAX});
        } else if (r <= Kb) {
            part = edge_row<TT, SAMPLE>(p, sh, target_row(tgt, b, K, V, r), ri, r, Kb, V, c, lane, cluster, CS, x_reg);
        } else {
            part = edge_row<TD, SAMPLE>(p, sh, draft_row(drf, b, K, V, r - Kb - 1), ri, r, Kb, V, c, lane, cluster,
                                        CS, x_reg);
        }
        if (lane == 0) sh.edge_part[r] = part;
    }
}

template <typename TT, typename TD, int MS>
__global__ void __launch_bounds__(NTHREADS, 2) verify_logits_kernel(VerifyParams p) {
    constexpr bool CAN_SAMPLE = (MS & MS_SAMPLE) != 0, CAN_GREEDY = (MS & MS_GREEDY) != 0;
    extern __shared__ __align__(128) char ring[];
    __shared__ SeqShared sh;
    // The next call on the stream may launch as soon as every CTA of this one
    // has started (its stores still wait for this one to complete): first
    // thing, so that consecutive calls launch at the hardware's pace rather
    // than one prologue apart.
    launch_dependents();
    cluster_arrive_started();
    cg::cluster_group cluster = cg::this_cluster();
    const int CS = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // A call may be launched with programmatic stream serialization, and then
    // start while the work ahead of it on the stream is finishing. A plain
    // call (no overlap flag, not the LM-head path) reads no input before that
    // work has completed: it waits here when its prologue reads inputs
    // (per-sequence modes or draft counts), otherwise just before its first
    // input read, once the input-free prologue has run. (Without the launch
    // attribute the wait returns at once.)
    const bool fused = p.target_parts != nullptr;
    const bool plain = !p.overlap_previous && !fused;
    const bool prologue_reads = p.modes != nullptr || p.draft_lens != nullptr;
    if (plain && prologue_reads) grid_dependency_wait();
    // Cluster c verifies sequence c, or, with per-sequence modes, the c-th of
    // the order (sample sequences, then the others, each in index order): the
    // sequences with the most rows to read start first. Every CTA derives the
    // same order from the modes array; results do not depend on it.
    if (warp == 0) {
        const int c = (int)(blockIdx.x / CS);
        int seq = c;
        if (p.modes && p.B <= MAX_ORDERED_B) {
            constexpr int PER = MAX_ORDERED_B / 32;
            unsigned smask[PER];
            int ns = 0;
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const int i = k * 32 + lane;
                const bool s = i < p.B && ld_in(p, p.modes + i, 0) == 1;
                smask[k] = __ballot_sync(FULL, s);
                ns += __popc(smask[k]);
            }
            const bool want_sample = c < ns;
            int left = want_sample ? c : c - ns;
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const int n_here = min(32, p.B - k * 32);
                unsigned m = want_sample ? smask[k] : (~smask[k] & (n_here >= 32 ? FULL : ((1u << max(n_here, 0)) - 1u)));
                const int cnt = __popc(m);
                if (left >= 0 && left < cnt) {
                    for (int t = 0; t < left; ++t) m &= m - 1u;
                    seq = k * 32 + __ffs(m) - 1;
                }
                left -= cnt;
            }
        }
        if (lane == 0) sh.seq_b = seq;
    }
    __syncthreads();
    const int b = sh.seq_b;
    const int K = p.K, V = p.V;
    const TT* tgt = static_cast<const TT*>(p.target);
    const TD* drf = static_cast<const TD*>(p.draft);

    // With overlap, the whole call may run alongside the work ahead of it,
    // and each thread that stores to global memory first waits for that work
    // to complete, just before its stores.
    const int mode = p.modes ? ld_in(p, p.modes + b, -1) : p.mode;
    // Kb: the drafts this sequence verifies (continuous batching), 0..K
    const int Kb = p.draft_lens ? ld_in(p, p.draft_lens + b, -1) : K;
    const bool len_ok = Kb >= 0 && Kb <= K;
    const bool mode_ok = (mode == 0 || mode == 1) && !(mode == 1 && drf == nullptr) && len_ok;
    const bool sample = CAN_SAMPLE && (!CAN_GREEDY || mode == 1) && mode_ok;
    // which partials this launch merges (a constant unless the set is mixed)
    const bool use_soft = !CAN_GREEDY || (CAN_SAMPLE && sample);
    const int nrows = mode_ok ? (sample ? 2 * Kb + 1 : Kb + 1) : 0;
    const float c = p.c;

    if (tid == 0) {
        for (int s = 0; s < NSTAGE; ++s) mbar_init(&sh.full[s], 1);
        mbar_init(&sh.never, 1);
        sh.err = 0;
        sh.total_chunks = 0;
        fence_barrier_init();
    }
    // (LM-head path: the target rows, and the draft rows when their partials
    // come from the GEMM too, take no pass-1 chunks and no edge slots)
    const bool fused_d = fused && p.draft_parts != nullptr;
    if (mode_ok && tid < nrows)
        sh.rows[tid] = (tid <= Kb ? fused : fused_d)
                           ? RowInfo{nullptr, 0, 0, 0, -1, -1, 0}
                           : tid <= Kb ? make_row_info<TT>(target_row(tgt, b, K, V, tid), V, rank, CS)
                                       : make_row_info<TD>(draft_row(drf, b, K, V, tid - Kb - 1), V, rank, CS);
    for (int t = tid; t < NCW * MAX_ROWS; t += NTHREADS) {
        const int w = t / MAX_ROWS, r = t % MAX_ROWS;
        sh.warp_part[w][r] = use_soft ? pack(SoftPart{-INFINITY, 0.0f}) : pack(ArgPart{-INFINITY, INT_MAX});
    }
    __syncthreads();
    if (mode_ok && warp == 0) {
        // prefix sums of the rows' chunk counts (the pass-1 schedule)
        int cnt = 0;
        for (int r0 = 0; r0 < nrows; r0 += 32) {
            const int r = r0 + lane;
            const int m = r < nrows ? (sh.rows[r].ib - sh.rows[r].ia + STAGE_SLOTS - 1) / STAGE_SLOTS : 0;
            int incl = m;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(FULL, incl, o);
                if (lane >= o) incl += y;
            }
            if (r < nrows) sh.rows[r].c1 = cnt + incl;
            cnt += __shfl_sync(FULL, incl, 31);
        }
        if (lane == 0) sh.total_chunks = cnt;
    }
    __syncthreads();
    const int total_chunks = mode_ok ? sh.total_chunks : 0;

    WarpRing wr{warp, 0u, 0u};
    uint32_t seq = 0;  // chunks this warp has handled, over both passes
    if (plain && !prologue_reads) grid_dependency_wait();  // the first input read follows
    // Lane i of every warp holds draft token x_i (first used after the
    // warp's first chunk has arrived, so the load overlaps the copies).
    const int x_reg = p.tree_parents ? (lane <= K ? ld_in(p, p.tokens + (size_t)b * (K + 1) + lane, -1) : -1)
                                     : (mode_ok && lane < Kb) ? ld_in(p, p.tokens + (size_t)b * K + lane, -1) : -1;

    // Pass 1 writes the captured logits into every CTA of the cluster.
    cluster_wait_started();

    // ---------------- pass 1: row partials over this CTA's slice ----------------
    // Warp 0 draws the Philox uniforms of positions 0..K while its first
    // copies are in flight; the decision reads them from shared memory.
    const uint64_t seqid = (sample && warp == 0 && p.seq_ids) ? ld_in(p, p.seq_ids + b, (uint64_t)b) : (uint64_t)b;
    auto draw_uniforms = [&] {
        if (warp == 0 && lane <= Kb) position_uniforms(p.seed, seqid, (uint32_t)lane, sh.u_pos[lane], sh.u2_pos[lane]);
    };
    if (mode_ok) {
        if constexpr (!CAN_GREEDY) {
            stream_pass1<TT, TD, true>(p, sh, wr, ring, total_chunks, nrows, c, warp, lane, seq, cluster, CS, Kb, x_reg, draw_uniforms);
        } else if constexpr (!CAN_SAMPLE) {
            stream_pass1<TT, TD, false>(p, sh, wr, ring, total_chunks, nrows, c, warp, lane, seq, cluster, CS, Kb, x_reg, [] {});
        } else {
            if (sample) stream_pass1<TT, TD, true>(p, sh, wr, ring, total_chunks, nrows, c, warp, lane, seq, cluster, CS, Kb, x_reg, draw_uniforms);
            else stream_pass1<TT, TD, false>(p, sh, wr, ring, total_chunks, nrows, c, warp, lane, seq, cluster, CS, Kb, x_reg, [] {});
        }
        if (warp == 0) {
            if constexpr (!CAN_GREEDY) {
                edge_pass1<TT, TD, true>(p, sh, tgt, drf, b, K, Kb, V, nrows, c, lane, cluster, CS, x_reg);
            } else if constexpr (!CAN_SAMPLE) {
                edge_pass1<TT, TD, false>(p, sh, tgt, drf, b, K, Kb, V, nrows, c, lane, cluster, CS, x_reg);
            } else {
                if (sample) edge_pass1<TT, TD, true>(p, sh, tgt, drf, b, K, Kb, V, nrows, c, lane, cluster, CS, x_reg);
                else edge_pass1<TT, TD, false>(p, sh, tgt, drf, b, K, Kb, V, nrows, c, lane, cluster, CS, x_reg);
            }
        }
    }
    // Failure-path tests: a bounded wait on a barrier that nothing completes
    // gives up exactly as a stalled copy's wait would.
    if (p.test_wait_timeout && tid == 0 && !mbar_wait(&sh.never, 0, 1u << 12)) atomicExch(&sh.err, 1);
    __syncthreads();
    // the draft logits at the draft tokens are inputs: read before the wait
    float ld_early = 0.0f;
    if (fused_d && sample && warp == 1 && lane < Kb && x_reg >= 0 && x_reg < V)
        ld_early = load_logit<TD>(p, draft_row(drf, b, K, V, lane), x_reg);
    if (fused) grid_dependency_wait();  // the GEMM grid ahead has completed; its stores are visible
    if (fused && mode_ok) {
        // the target logits at the draft tokens: in flight during the merge
        float lt_early = 0.0f;
        if constexpr (sizeof(TT) == 4) {
            if (sample && warp == 0 && lane < Kb && x_reg >= 0 && x_reg < V)
                lt_early = ldcg_in(p, target_row(tgt, b, K, V, lane) + x_reg, 0.0f);
        }
        // This CTA's share of every row computed by the GEMM is the merge of
        // its contiguous run of the GEMM CTAs' partials: lanes take every
        // 32nd one in order (four loads in flight), then a butterfly merges
        // the lanes (the merges are symmetric, so every lane ends with the
        // same bits).
        int t0, t1;
        split_range(p.part_tiles, rank, CS, t0, t1);
        const float2 empty = use_soft ? pack(SoftPart{-INFINITY, 0.0f}) : pack(ArgPart{-INFINITY, INT_MAX});
        const int n_fused = fused_d ? nrows : Kb + 1;
        const int Md = p.B * K;
        // a warp takes rows warp and warp + NCW together, so that both rows'
        // loads are in flight at once
        auto col_of = [&](int r, size_t& stride) -> const float2* {
            const bool tr = r <= Kb;
            stride = tr ? (size_t)p.part_M : (size_t)Md;
            return tr ? p.target_parts + (size_t)b * (K + 1) + r : p.draft_parts + (size_t)b * K + (r - Kb - 1);
        };
        auto merge2 = [&](float2 a, float2 c) -> float2 {
            return use_soft ? pack(merge_soft(as_soft(a), as_soft(c))) : pack(merge_arg(as_arg(a), as_arg(c)));
        };
        for (int r0 = warp; r0 < n_fused; r0 += 2 * NCW) {
            const int r1 = r0 + NCW;
            size_t s0, s1;
            const float2* c0 = col_of(r0, s0);
            const float2* c1 = r1 < n_fused ? col_of(r1, s1) : c0;
            if (r1 >= n_fused) s1 = s0;
            float2 acc0 = empty, acc1 = empty;
            for (int t = t0 + lane; t < t1; t += 4 * 32) {
                float2 v0[4], v1[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const bool in = t + 32 * u < t1;
                    v0[u] = in ? ldcg_in(p, c0 + (size_t)(t + 32 * u) * s0, empty) : empty;
                    v1[u] = in && r1 < n_fused ? ldcg_in(p, c1 + (size_t)(t + 32 * u) * s1, empty) : empty;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    acc0 = merge2(acc0, v0[u]);
                    acc1 = merge2(acc1, v1[u]);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                acc0 = merge2(acc0, make_float2(__shfl_xor_sync(FULL, acc0.x, o), __shfl_xor_sync(FULL, acc0.y, o)));
                acc1 = merge2(acc1, make_float2(__shfl_xor_sync(FULL, acc1.x, o), __shfl_xor_sync(FULL, acc1.y, o)));
            }
            if (lane == 0) {
                sh.edge_part[r0] = acc0;
                if (r1 < n_fused) sh.edge_part[r1] = acc1;
            }
        }
        // the logits at the draft tokens, for the decision (every CTA)
        if (sizeof(TT) == 4 && sample && warp == 0 && lane < Kb && x_reg >= 0 && x_reg < V) sh.lt_x[lane] = lt_early;
        if (fused_d && sample && warp == 1 && lane < Kb && x_reg >= 0 && x_reg < V) sh.ld_x[lane] = ld_early;
        __syncthreads();
    }
    // This CTA's partial of every row, pushed into every CTA of the cluster.
    for (int t = tid; mode_ok && t < CS * nrows; t += NTHREADS) {
        const int dst = t / nrows, r = t % nrows;
        float2 acc = sh.edge_part[r];
        for (int w = 0; w < NCW; ++w) {
            acc = use_soft ? pack(merge_soft(as_soft(acc), as_soft(sh.warp_part[w][r])))
                           : pack(merge_arg(as_arg(acc), as_arg(sh.warp_part[w][r])));
        }
        if (sh.err) acc = make_float2(__int_as_float(0x7fc00000), 0.0f);  // poison: invalid
        cluster.map_shared_rank(&sh.gathered[0][0], dst)[rank * MAX_ROWS + r] = acc;
    }
    cluster.sync();

    // Every row's CS partials merge in a butterfly over lanes: lane (r, cr) of
    // a row group holds CTA cr's partial of row r. The merge is symmetric, so
    // every CTA (and every lane) obtains the same bits.
    if (mode_ok) {
        const int rows_per_pass = 32 / CS;
        const int r_in = lane / CS, cr = lane % CS;
        const float2 empty = use_soft ? pack(SoftPart{-INFINITY, 0.0f}) : pack(ArgPart{-INFINITY, INT_MAX});
        for (int r0 = warp * rows_per_pass; r0 < nrows; r0 += NCW * rows_per_pass) {
            const int r = r0 + r_in;
            float2 acc = r < nrows ? sh.gathered[cr][r] : empty;
            for (int o = CS >> 1; o > 0; o >>= 1) {
                const float2 other = make_float2(__shfl_xor_sync(FULL, acc.x, o), __shfl_xor_sync(FULL, acc.y, o));
                acc = use_soft ? pack(merge_soft(as_soft(acc), as_soft(other)))
                               : pack(merge_arg(as_arg(acc), as_arg(other)));
            }
            if (cr == 0 && r < nrows) sh.merged[r] = acc;
        }
    }
    __syncthreads();

    // ---------------- decide (redundantly in every CTA) ----------------
    if (MS == MS_GREEDY && warp == 0 && p.tree_parents) {
        tree_decide(p, sh, b, K + 1, V, lane, rank, mode_ok, x_reg);
    } else if (warp == 0) {
        bool bad = !mode_ok;
        if (mode_ok) {
            for (int r = lane; r < nrows; r += 32) {
                const float2 acc = sh.merged[r];
                if (use_soft) {
                    const SoftPart sp = as_soft(acc);
                    bad |= !(isfinite(sp.R) && isfinite(sp.s) && sp.s > 0.0f);
                } else {
                    const ArgPart ap = as_arg(acc);
                    bad |= !isfinite(ap.v) || ap.i < 0 || ap.i >= V;
                }
            }
        }
        float u = 0.0f, u2 = 0.0f;
        if (sample && lane <= Kb) {
            u = sh.u_pos[lane];
            u2 = sh.u2_pos[lane];
        }
        int x = -1;
        bool bad_token = false, rej = false;
        float et = 0.0f, ed = 0.0f, St = 1.0f, Sd = 1.0f;
        if (mode_ok && lane < Kb) {
            x = x_reg;
            bad_token = x < 0 || x >= V;
            if (!bad_token && mode_ok) {
                if (!use_soft) {
                    rej = x != as_arg(sh.merged[lane]).i;
                } else {
                    const SoftPart st = as_soft(sh.merged[lane]);
                    const SoftPart sd = as_soft(sh.merged[Kb + 1 + lane]);
                    // the logits at x, captured during pass 1 by the CTA holding them
                    et = ex2(fmaf(sh.lt_x[lane], c, -st.R));
                    ed = ex2(fmaf(sh.ld_x[lane], c, -sd.R));
                    St = st.s;
                    Sd = sd.s;
                    rej = !accept_draft(u, ed, St, et, Sd);
                }
            }
        }
        const bool any_bad_token = __any_sync(FULL, bad_token);
        const bool invalid = __any_sync(FULL, bad) || any_bad_token;
        const unsigned rejm = __ballot_sync(FULL, rej);
        const int j = rejm ? __ffs(rejm) - 1 : Kb;
        const float u2j = __shfl_sync(FULL, u2, j);
        if (lane == 0) {
            sh.j = j;
            sh.valid = !invalid;
            sh.sample = sample;
            sh.u2 = u2j;
            if (sample && !invalid) {
                sh.st = as_soft(sh.merged[j]);
                sh.use_d = j < Kb;
                sh.sd = j < Kb ? as_soft(sh.merged[Kb + 1 + j]) : SoftPart{-INFINITY, 0.0f};
            }
        }
        // With overlap, a call that goes on to pass 2 stores this row at its
        // very end instead (where its stores wait for the previous call), so
        // that waiting holds up none of its own work.
        if (rank == 0 && !(p.overlap_previous && sample && !invalid)) {
            if (p.overlap_previous) grid_dependency_wait();  // the stores below follow the previous call's
            const int greedy_tok = (!sample && !invalid) ? as_arg(sh.merged[j]).i : -1;
            if (lane <= K) {
                int tok = -1;
                if (!invalid) tok = lane < j ? x : (lane == j ? greedy_tok : -1);
                // in sample mode position j belongs to the CTA that finds the draw
                if (!(sample && !invalid && lane == j))
                    st_out(p, p.out_tokens + ((size_t)b * (K + 1) + lane), tok);
            }
            if (lane == 0) st_out(p, p.out_n_accepted + (b), invalid ? -1 : j);
            if (lane < K) {
                const float qnan = __int_as_float(0x7fc00000);
                const bool tested = sample && !invalid && lane < Kb;
                if (p.out_p_target) st_out(p, p.out_p_target + ((size_t)b * K + lane), tested ? et / St : qnan);
                if (p.out_p_draft) st_out(p, p.out_p_draft + ((size_t)b * K + lane), tested ? ed / Sd : qnan);
            }
            if (lane == 0 && (!sample || invalid) && p.out_residual_mass)
                st_out(p, p.out_residual_mass + (b), __int_as_float(0x7fc00000));
            if (lane < 2 && (!sample || invalid) && p.out_draw_edges)
                st_out(p, p.out_draw_edges + (2 * (size_t)b + lane), __int_as_float(0x7fc00000));
            if (lane == 0 && p.status_word && invalid)
                atomicOr(p.status_word, !len_ok        ? (unsigned)SV_FLAG_BAD_LENGTH
                                        : !mode_ok     ? (unsigned)SV_FLAG_BAD_MODE
                                        : any_bad_token ? (unsigned)SV_FLAG_BAD_TOKEN
                                                        : (unsigned)SV_FLAG_BAD_ROW);
            if (lane == 0 && p.status_word && sh.err) atomicOr(p.status_word, (unsigned)SV_FLAG_TIMEOUT);
        }
    }
    __syncthreads();

    if (!CAN_SAMPLE || !(sh.sample && sh.valid)) {
        wr.drain(sh);
        return;  // every remote access of this CTA's shared memory happened before the barrier
    }

    // ---------------- pass 2: mass of the final draw over row j ----------------
    const int j = sh.j;
    DrawSrc<TT, TD> src;
    src.trow = tgt + ((size_t)b * (K + 1) + j) * V;
    src.drow = sh.use_d ? drf + ((size_t)b * K + j) * V : reinterpret_cast<const TD*>(src.trow);
    src.gt = row_geom(src.trow, V);
    src.gd = row_geom(src.drow, V);
    src.V = V;
    src.same_slots = std::is_same<TT, TD>::value && src.gd.head == src.gt.head;
    int qa, qb;
    split_range(src.gt.nslot, rank, CS, qa, qb);
    const WarpSlots sl = warp_slots<TT>(src.gt, V, qa, qb);
    const bool draft_in_ring = src.same_slots;
    // bf16 draft under fp32 target: the draft streams as the aligned span of
    // each chunk's elements (8 bytes per target slot, at most 1040 of the
    // stage's 2048-byte draft half)
    constexpr bool SPAN_TYPES = sizeof(TT) == 4 && sizeof(TD) == 2;
    static_assert(!SPAN_TYPES || 8 * P2_SLOTS + 16 <= STAGE_BYTES - P2_DRAFT_OFF, "draft span must fit");
    const uint32_t span_off = SPAN_TYPES ? draft_span<TT, TD>(src, sl.ia, 0).off : 0u;
    DrawRows w;
    w.c = c;
    w.ntR = -sh.st.R;
    w.invSt = 1.0f / sh.st.s;
    w.ndR = -sh.sd.R;
    w.invSd = sh.use_d ? 1.0f / sh.sd.s : 0.0f;
    pack_draw_rows(w);
    const int n_chunks = (sl.ib - sl.ia + P2_SLOTS - 1) / P2_SLOTS;
    constexpr int STEPS = P2_SLOTS / 32;

    // When pass 1's chunks all fit the ring (none was refilled), chunk c still
    // sits in stage c, so row r's interior slot q is at ring + 16 (c0 *
    // STAGE_SLOTS + q - ia): row j's slices are read back from shared memory
    // instead of HBM.
    const RowInfo rt = sh.rows[j];
    const bool resident_t = !fused && total_chunks <= NSTAGE && rt.ia == sl.ia && rt.ib == sl.ib;
    const int rd_row = sh.use_d ? Kb + 1 + j : j;
    const RowInfo rd = sh.rows[rd_row];
    const int rt_c0 = row_c0(sh.rows, j), rd_c0 = row_c0(sh.rows, rd_row);
    const bool resident_d = resident_t && draft_in_ring && rd.ia == sl.ia && rd.ib == sl.ib;
    int attempt = 0;
    bool fell_back = false;
    bool last_resident = false;  // the last attempt read row j from pass 1's stages
    for (;; ++attempt) {
        w.use_d = sh.use_d && attempt == 0;
        const bool ring_d = w.use_d && draft_in_ring;
        const bool span_d = SPAN_TYPES && w.use_d;
        const bool resident = resident_t && (!ring_d || resident_d) && !span_d;
        last_resident = resident;
        if (lane == 0) sh.p2_seq0[warp] = (unsigned char)(seq % NBUF);
        if (!sh.err) {
            for (int jj = 0; !resident && jj < NBUF; ++jj) {
                const int ci = warp + NCW * jj;
                if (ci < n_chunks) fill_pass2<TT, TD>(p, sh, wr, ring, seq + jj, src, sl.ia, sl.ib, ci, ring_d, span_d, lane);
            }
            for (int ci = warp; ci < n_chunks; ci += NCW) {
                const int q = sl.ia + ci * P2_SLOTS;
                const int n = min(P2_SLOTS, sl.ib - q);
                uint4 dt[STEPS], dd[STEPS];
                if (resident) {
                    const char* res_t = ring + (size_t)(rt_c0 * STAGE_SLOTS + ci * P2_SLOTS) * 16;
                    const char* res_d = ring + (size_t)(rd_c0 * STAGE_SLOTS + ci * P2_SLOTS) * 16;
#pragma unroll
                    for (int kk = 0; kk < STEPS; ++kk) {
                        const int i = kk * 32 + lane;
                        dt[kk] = i < n ? lds128(res_t + i * 16) : neg_inf_slot<TT>();
                        dd[kk] = (ring_d && i < n) ? lds128(res_d + i * 16) : neg_inf_slot<TT>();
                    }
                } else {
                    if (!wr.wait(sh, seq)) {
                        atomicExch(&sh.err, 1);
                        break;
                    }
                    const char* stage = wr.stage(ring, seq);
#pragma unroll
                    for (int kk = 0; kk < STEPS; ++kk) {
                        const int i = kk * 32 + lane;
                        dt[kk] = neg_inf_slot<TT>();
                        dd[kk] = neg_inf_slot<TT>();
                        if (i < n) {
                            dt[kk] = lds128(stage + i * 16);
                            if (ring_d) dd[kk] = lds128(stage + P2_DRAFT_OFF + i * 16);
                            if (span_d) dd[kk] = span_slot(stage + P2_DRAFT_OFF, span_off, i);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (ci + NBUF * NCW < n_chunks)
                        fill_pass2<TT, TD>(p, sh, wr, ring, seq + NBUF, src, sl.ia, sl.ib, ci + NBUF * NCW, ring_d, span_d,
                                           lane);
                    ++seq;
                }
                // the chunk's draw mass: per lane over its slots, then one warp sum
                f32x2 acc = 0ull;
#pragma unroll
                for (int kk = 0; kk < STEPS; ++kk) {
                    const int i = kk * 32 + lane;
                    if (w.use_d && !draft_in_ring && !span_d && i < n)
                        dd[kk] = load_elems_as<TT, TD>(p, src.drow, V, (q + i) * Elem<TT>::E - src.gt.head);
#pragma unroll
                    for (int k2 = 0; k2 < Elem<TT>::E / 2; ++k2)
                        acc = add2(acc, draw_mass2(w, slot_pair<TT>(dt[kk], k2), slot_pair<TT>(dd[kk], k2)));
                }
                float a0, a1;
                unpack2(acc, a0, a1);
                float part = a0 + a1;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(FULL, part, o);
                if (lane == 0) sh.p2_part[ci] = part;
            }
        }
        if (warp == 0) {
            // the partial slots at the two ends of this CTA's slice
            float e_lo = 0.0f, e_hi = 0.0f;
            if (sl.edge_lo >= 0 || sl.edge_hi >= 0) {
                uint4 dt, dd;
                const int q = lane == 0 ? sl.edge_lo : lane == 1 ? sl.edge_hi : -1;
                load_draw_slot<TT, TD>(p, src, w.use_d, q, dt, dd);
                const float m = slot_mass<TT>(w, dt, dd);
                e_lo = __shfl_sync(FULL, m, 0);
                e_hi = __shfl_sync(FULL, m, 1);
            }
            if (lane == 0) {
                sh.p2_edge[0] = e_lo;
                sh.p2_edge[1] = e_hi;
            }
        }
        __syncthreads();
        // this CTA's draw mass (float-float), pushed to every CTA
        if (warp == 0) {
            ff t = ff_from(0.0f);
            for (int i = lane; i < n_chunks; i += 32) t = ff_add(t, sh.p2_part[i]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) t = ff_add(t, ff_shfl_xor(t, o));
            t = ff_add(ff_add(t, sh.p2_edge[0]), sh.p2_edge[1]);
            if (sh.err) t = ff_from(0.0f);
            t = ff_shfl(t, 0);  // one value for every destination CTA
            if (lane < CS) cluster.map_shared_rank(&sh.gathered_tot[0][0], lane)[attempt * MAX_CS + rank] = make_float2(t.hi, t.lo);
        }
        cluster.sync();
        // the cluster's total and, for the draw, the CTA whose mass holds
        // t = u2 * total: an inclusive float-float scan over lanes cr < CS
        if (warp == 0) {
            const float2 g = lane < CS ? sh.gathered_tot[attempt][lane] : make_float2(0.0f, 0.0f);
            const ff v{g.x, g.y};
            ff incl = v;
#pragma unroll
            for (int o = 1; o < MAX_CS; o <<= 1) {
                const ff y = ff_shfl_up(incl, o);
                if (lane >= o) incl = ff_add(y, incl);
            }
            const ff S = ff_shfl(incl, MAX_CS - 1);
            const ff t = ff_mul(S, sh.u2);
            const unsigned hit = __ballot_sync(FULL, lane < CS && ff_gt(incl, t));
            const unsigned pos = __ballot_sync(FULL, lane < CS && v.hi > 0.0f);
            const ff excl = ff_add(incl, ff_neg(v));
            int cstar;
            ff tc;
            if (hit) {
                cstar = __ffs(hit) - 1;
                tc = ff_shfl(ff_add(t, ff_neg(excl)), cstar);
            } else {  // t at or past the summed mass: take the last positive element
                cstar = pos ? 31 - __clz(pos) : -1;
                tc = ff{INFINITY, 0.0f};
            }
            if (lane == 0) {
                sh.total = S;
                sh.cstar = cstar;
                sh.tc = tc;
            }
        }
        __syncthreads();
        if (sh.total.hi > 0.0f || !w.use_d) break;
        // The residual summed to zero in float: fall back to P_t of row j
        // (reported at the end).
        fell_back = true;
    }


    if (rank == sh.cstar) {  // the CTA holding the draw (uniform over the CTA)
        if (warp == 0) {
            // Walk down this CTA's parts in index order (low edge slot, the
            // chunk parts, high edge slot): each lane sums a contiguous run of
            // parts, a warp scan finds the run holding tc, its lane walks it.
            const int P = n_chunks + 2;
            auto part_val = [&](int i) -> float {
                if (i == 0) return sh.p2_edge[0];
                if (i == P - 1) return sh.p2_edge[1];
                return sh.p2_part[i - 1];
            };
            const int per = (P + 31) / 32;
            const int i0 = min(P, lane * per), i1 = min(P, i0 + per);
            ff mine = ff_from(0.0f);
            int last_pos = -1;
            for (int i = i0; i < i1; ++i) {
                const float v = part_val(i);
                mine = ff_add(mine, v);
                if (v > 0.0f) last_pos = i;
            }
            ff incl = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const ff y = ff_shfl_up(incl, o);
                if (lane >= o) incl = ff_add(y, incl);
            }
            const ff tc = sh.tc;
            const bool tc_inf = isinf(tc.hi);
            const unsigned hit = __ballot_sync(FULL, !tc_inf && ff_gt(incl, tc));
            int found = -1;
            ff tw{INFINITY, 0.0f};
            if (hit) {
                const int l = __ffs(hit) - 1;
                if (lane == l) {
                    ff t = ff_add(tc, ff_neg(ff_add(incl, ff_neg(mine))));
                    for (int i = i0; i < i1; ++i) {
                        const float v = part_val(i);
                        if (ff_gt(ff_from(v), t)) { found = i; tw = t; break; }
                        t = ff_add(t, -v);
                    }
                    if (found < 0) found = last_pos;  // rounding: this run's last positive part
                }
                found = __shfl_sync(FULL, found, l);
                tw = ff_shfl(tw, l);
            }
            if (found < 0) {  // rounding put tc past every part: the last positive part
                int lp = last_pos;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(FULL, lp, o));
                found = lp;
                tw = ff{INFINITY, 0.0f};
            }
            if (lane == 0) {
                sh.found = found;
                sh.tw = tw;
            }
        }
        __syncthreads();
        // Inverse CDF inside the part: warp k takes its k-th step of 32 slots
        // (all loaded at once); the first step whose running mass passes tw
        // holds the token.
        const int found = sh.found;
        constexpr int STEPS = P2_SLOTS / 32;
        if (found >= 0) {
            const int P = n_chunks + 2;
            int q0, n;
            if (found == 0) { q0 = sl.edge_lo; n = 1; }
            else if (found == P - 1) { q0 = sl.edge_hi; n = 1; }
            else {
                q0 = sl.ia + (found - 1) * P2_SLOTS;
                n = min(P2_SLOTS, sl.ib - q0);
            }
            const ff tw = sh.tw;
            const bool tw_inf = isinf(tw.hi);
            // The part's chunk may still be in shared memory: in pass 1's
            // stages (row j read back from them), or in the stage pass 2 copied
            // it to when no stage was refilled (at most NSTAGE chunks).
            const bool interior = found > 0 && found < P - 1 && !sh.err;
            const char* at_t = nullptr;
            const char* at_d = nullptr;
            if (interior && last_resident) {
                at_t = ring + (size_t)(rt_c0 * STAGE_SLOTS + (found - 1) * P2_SLOTS) * 16;
                at_d = ring + (size_t)(rd_c0 * STAGE_SLOTS + (found - 1) * P2_SLOTS) * 16;
            } else if (interior && n_chunks <= NSTAGE) {
                const int ci = found - 1, wc = ci % NCW;
                at_t = ring + (size_t)(wc + NCW * ((sh.p2_seq0[wc] + ci / NCW) % NBUF)) * STAGE_BYTES;
                at_d = at_t + P2_DRAFT_OFF;
            }
            DrawStep<TT, TD> st;
            if (warp < STEPS) {
                if (at_t) {
                    const int i = warp * 32 + lane;
                    const int q = i < n ? q0 + i : -1;
                    uint4 dt = neg_inf_slot<TT>(), dd = neg_inf_slot<TT>();
                    if (i < n) {
                        dt = lds128(at_t + i * 16);
                        if (w.use_d && draft_in_ring) dd = lds128(at_d + i * 16);
                        else if (SPAN_TYPES && w.use_d && !last_resident) dd = span_slot(at_d, span_off, i);
                        else if (w.use_d) dd = load_elems_as<TT, TD>(p, src.drow, V, q * Elem<TT>::E - src.gt.head);
                    }
                    st.take(w, dt, dd, q, src.gt.head, lane);
                } else {
                    st.load(p, src, w, q0, n, warp, lane);
                }
                if (lane == 0) {
                    sh.step_tot[warp] = st.tot;
                    sh.step_lp[warp] = st.last_pos;
                }
            }
            __syncthreads();
            ff run = ff_from(0.0f);
            if (warp < STEPS) {
                for (int k = 0; k < warp; ++k) run = ff_add(run, sh.step_tot[k]);
                const unsigned hit = __ballot_sync(FULL, !tw_inf && ff_gt(ff_add(run, st.incl), tw));
                if (lane == 0) sh.step_hit[warp] = hit ? __ffs(hit) - 1 : -1;
            }
            __syncthreads();
            int kstar = -1;
            for (int k = STEPS - 1; k >= 0; --k)
                if (sh.step_hit[k] >= 0) kstar = k;
            if (kstar >= 0 && warp == kstar) {
                const int l = sh.step_hit[kstar];
                float d0, d1;
                const int token = st.walk(run, tw, l, d0, d1);
                if (lane == l) {
                    if (p.overlap_previous) grid_dependency_wait();
                    st_out(p, p.out_tokens + ((size_t)b * (K + 1) + j), token);
                    if (p.out_draw_edges) {
                        st_out(p, p.out_draw_edges + (2 * (size_t)b), d0);
                        st_out(p, p.out_draw_edges + (2 * (size_t)b + 1), d1);
                    }
                }
            } else if (kstar < 0 && tid == 0) {
                int lp = -1;  // tw past the part's mass: its last positive element
                for (int k = 0; k < STEPS; ++k) lp = max(lp, sh.step_lp[k]);
                if (p.overlap_previous) grid_dependency_wait();
                st_out(p, p.out_tokens + ((size_t)b * (K + 1) + j), lp);
                if (p.out_draw_edges) {
                    st_out(p, p.out_draw_edges + (2 * (size_t)b), 0.0f);
                    st_out(p, p.out_draw_edges + (2 * (size_t)b + 1), 0.0f);
                }
            }
        }
    }

    // Rank 0's row and flags, after the previous call's stores when calls overlap.
    if (rank == 0 && warp == 0) {
        if (p.overlap_previous) {
            grid_dependency_wait();
            // the decision's stores, deferred from the decide step (lanes
            // other than j; position j is the draw's)
            if (lane <= K && lane != j) st_out(p, p.out_tokens + ((size_t)b * (K + 1) + lane), lane < j ? x_reg : -1);
            if (lane == 0) st_out(p, p.out_n_accepted + (b), j);
            if (lane < K && (p.out_p_target || p.out_p_draft)) {
                const float qnan = __int_as_float(0x7fc00000);
                float pt = qnan, pd = qnan;
                if (lane < Kb) {
                    const SoftPart st = as_soft(sh.merged[lane]);
                    const SoftPart sd = as_soft(sh.merged[Kb + 1 + lane]);
                    pt = ex2(fmaf(sh.lt_x[lane], c, -st.R)) / st.s;
                    pd = ex2(fmaf(sh.ld_x[lane], c, -sd.R)) / sd.s;
                }
                if (p.out_p_target) st_out(p, p.out_p_target + ((size_t)b * K + lane), pt);
                if (p.out_p_draft) st_out(p, p.out_p_draft + ((size_t)b * K + lane), pd);
            }
            if (lane == 0 && p.status_word && sh.err) atomicOr(p.status_word, (unsigned)SV_FLAG_TIMEOUT);
        }
        if (lane == 0) {
            if (p.status_word && fell_back) atomicOr(p.status_word, (unsigned)SV_FLAG_RESIDUAL_FALLBACK);
            if (sh.cstar >= 0 && isinf(sh.tc.hi) && p.status_word)
                atomicOr(p.status_word, (unsigned)SV_FLAG_DRAW_EDGE);
            if (sh.cstar < 0) {
                // No mass at all (cannot happen for a valid row): report the
                // sequence as invalid rather than leave a slot unwritten.
                st_out(p, p.out_tokens + ((size_t)b * (K + 1) + j), -1);
                st_out(p, p.out_n_accepted + (b), -1);
                if (p.out_draw_edges) {
                    st_out(p, p.out_draw_edges + (2 * (size_t)b), __int_as_float(0x7fc00000));
                    st_out(p, p.out_draw_edges + (2 * (size_t)b + 1), __int_as_float(0x7fc00000));
                }
                if (p.status_word) atomicOr(p.status_word, (unsigned)SV_FLAG_BAD_ROW);
            }
            if (p.out_residual_mass) st_out(p, p.out_residual_mass + (b), sh.total.hi + sh.total.lo);
        }
    }
    wr.drain(sh);
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
// Type pairs (target, draft): 0 = fp32/fp32, 1 = bf16/bf16, 2 = fp32/bf16.
constexpr int N_COMBOS = 3;

// Dynamic shared memory of a launch whose clusters fit on the GPU at one CTA
// per SM: the kernel uses RING_BYTES of it; the rest keeps a second CTA off
// the SM, so a small batch spreads over twice as many SMs.
constexpr int SPREAD_SMEM = 128 * 1024;

// Function attributes are per device; set them once per device, pair and
// mode set (index MS - 1).
static std::atomic<int> g_attr_done[64][N_COMBOS][3];

template <typename TT, typename TD>
static constexpr int combo_of() {
    return std::is_same<TT, TD>::value ? (sizeof(TT) == 4 ? 0 : 1) : 2;
}

template <typename TT, typename TD, int MS>
static cudaError_t prepare_kernel() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    constexpr int ci = combo_of<TT, TD>();
    if (dev >= 0 && dev < 64 && g_attr_done[dev][ci][MS - 1].load(std::memory_order_acquire)) return cudaSuccess;
    e = cudaFuncSetAttribute(verify_logits_kernel<TT, TD, MS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SPREAD_SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(verify_logits_kernel<TT, TD, MS>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) g_attr_done[dev][ci][MS - 1].store(1, std::memory_order_release);
    return cudaSuccess;
}

static void fill_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, unsigned grid, int cs,
                        cudaStream_t stream, int smem) {
    cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
}

template <typename TT, typename TD, int MS>
static int max_active_clusters(int cs, int smem = RING_BYTES) {
    if (prepare_kernel<TT, TD, MS>() != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    fill_config(cfg, attr, (unsigned)cs, cs, 0, smem);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, verify_logits_kernel<TT, TD, MS>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// Per device, pair, mode set and log2(cluster size): how many clusters are
// co-resident at one CTA per SM, plus one (0 = not yet known); the SM count.
static std::atomic<int> g_spread_clusters[64][N_COMBOS][3][5];
static std::atomic<int> g_num_sms[64];

static int log2_cs(int cs) { return cs >= 16 ? 4 : cs >= 8 ? 3 : cs >= 4 ? 2 : cs >= 2 ? 1 : 0; }

// One CTA per SM when every cluster of the launch is co-resident that way.
template <typename TT, typename TD, int MS>
static int launch_smem(int B, int cs) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return RING_BYTES;
    int sms = g_num_sms[dev].load(std::memory_order_acquire);
    if (sms == 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return RING_BYTES;
        }
        g_num_sms[dev].store(sms, std::memory_order_release);
    }
    if ((long long)B * cs > sms) return RING_BYTES;
    std::atomic<int>& slot = g_spread_clusters[dev][combo_of<TT, TD>()][MS - 1][log2_cs(cs)];
    int n = slot.load(std::memory_order_acquire);
    if (n == 0) {
        n = max_active_clusters<TT, TD, MS>(cs, SPREAD_SMEM) + 1;
        slot.store(n, std::memory_order_release);
    }
    return n - 1 >= B ? SPREAD_SMEM : RING_BYTES;
}

template <typename TT, typename TD, int MS>
static cudaError_t launch_ms(const VerifyParams& p, int cs, cudaStream_t stream) {
    cudaError_t e = prepare_kernel<TT, TD, MS>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    // Calls that overlap the previous one share the GPU with it: two CTAs
    // per SM let more calls' copies be in flight at once (c2 back to back:
    // 2.94 -> 2.70 us per call on GB300); a lone call spreads out instead.
    const int smem = p.overlap_previous ? RING_BYTES : launch_smem<TT, TD, MS>(p.B, cs);
    fill_config(cfg, attr, (unsigned)(p.B * cs), cs, stream, smem);
    // The call may launch before the work ahead of it has completed; the
    // kernel waits for that work before its first input read (plain calls)
    // or first store (overlap). Plain calls do so only when their grid
    // spreads one CTA per SM: a larger grid whose CTAs took SMs one by one as
    // the previous grid's left ended up worse placed than one launched onto
    // an idle GPU (measured on GB300: c3 37.6 -> 42.4 us, c4 235 -> 240 us;
    // c2, spread, 14.6 -> 13.1 us).
    if (p.overlap_previous || p.target_parts || smem == SPREAD_SMEM) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, verify_logits_kernel<TT, TD, MS>, p);
}

// The mode set a launch needs: trees and all-greedy batches run the greedy
// kernel, all-sample batches the sample kernel, per-sequence modes both.
template <typename TT, typename TD>
static cudaError_t launch_typed(const VerifyParams& p, int cs, cudaStream_t stream) {
    if (p.tree_parents || (!p.modes && p.mode == SV_GREEDY)) return launch_ms<TT, TD, MS_GREEDY>(p, cs, stream);
    if (!p.modes && p.mode == SV_SAMPLE) return launch_ms<TT, TD, MS_SAMPLE>(p, cs, stream);
    return launch_ms<TT, TD, MS_MIXED>(p, cs, stream);
}

static int combo_index(int dtype_target, int dtype_draft) {
    if (dtype_target == SV_F32 && dtype_draft == SV_F32) return 0;
    if (dtype_target == SV_BF16 && dtype_draft == SV_BF16) return 1;
    if (dtype_target == SV_F32 && dtype_draft == SV_BF16) return 2;
    return -1;
}

bool supported_dtypes(int dtype_target, int dtype_draft) {
    return combo_index(dtype_target, dtype_draft) >= 0;
}

// Per device, type pair and log2(cluster size): 0 unknown, 1 usable, 2 not.
static std::atomic<int> g_cluster_ok[64][N_COMBOS][5];

int usable_cluster_size(int dtype_target, int dtype_draft, int cs) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    const int ci = combo_index(dtype_target, dtype_draft);
    if (ci < 0) return 0;
    for (; cs >= 1; cs >>= 1) {
        const int lg = log2_cs(cs);
        int state = g_cluster_ok[dev][ci][lg].load(std::memory_order_acquire);
        if (state == 0) {
            const int n = ci == 0   ? max_active_clusters<float, float, MS_MIXED>(cs)
                          : ci == 1 ? max_active_clusters<__nv_bfloat16, __nv_bfloat16, MS_MIXED>(cs)
                                    : max_active_clusters<float, __nv_bfloat16, MS_MIXED>(cs);
            state = n > 0 ? 1 : 2;
            g_cluster_ok[dev][ci][lg].store(state, std::memory_order_release);
        }
        if (state == 1) return cs;
    }
    return 0;
}

int min_cluster_size(int V, int esize) {
    const long long nslot = ((long long)V * esize + 15) / 16 + 1;
    if (nslot > (1LL << 26)) return 0;  // keeps the slot arithmetic inside 32 bits
    const long long cap = (long long)MAX_P2_CHUNKS * P2_SLOTS;  // slots per CTA slice
    int cs = 1;
    while (cs < MAX_CS && (nslot + cs - 1) / cs > cap) cs *= 2;
    return (nslot + cs - 1) / cs > cap ? 0 : cs;
}

// The smallest power of two that gives every SM a CTA, while each CTA keeps at
// least two chunks of every row (measured best on GB300 for the workloads).
int auto_cluster_size(int B, int V, int esize, int num_sms) {
    const long long nslot = ((long long)V * esize + 15) / 16;
    int cs = 1;
    while (cs < MAX_CS && (long long)B * cs < num_sms && nslot / (2LL * cs) >= STAGE_SLOTS) cs *= 2;
    const int lo = min_cluster_size(V, esize);
    return cs < lo ? lo : cs;
}

// For calls that overlap the previous one: one CTA per sequence. Consecutive
// overlapping calls finish one after another (each stores only once the
// previous call has completed, about 2 us per call), so what sets the rate is
// how many calls' copies are in flight: few CTAs per call, two per SM, let
// many calls run at once. Measured best on GB300 against clusters of 2-8 for
// B=8 x 11 rows of 32000 fp32 and B=64 x (5 or 9) rows of 128256 bf16
// (22.3 us per call against 26.1 us with clusters of 4).
int overlap_cluster_size() { return 1; }

// For the LM-head path, whose verify streams only the final draw's rows: the
// largest power of two (at most 8) that keeps every CTA of the launch on its
// own SM. Its CTAs may start while the GEMM's last CTAs run; clusters of 8
// placed then left later clusters without room until the first ones ended
// (measured on GB300 for B = 32), which one CTA per SM avoids.
int fused_cluster_size(int B, int num_sms) {
    int cs = 1;
    while (cs < 8 && (long long)B * cs * 2 <= num_sms) cs *= 2;
    return cs;
}

cudaError_t launch_verify_logits(const VerifyParams& p, int dtype_target, int dtype_draft, int cs,
                                 cudaStream_t stream) {
    switch (combo_index(dtype_target, dtype_draft)) {
        case 0: return launch_typed<float, float>(p, cs, stream);
        case 1: return launch_typed<__nv_bfloat16, __nv_bfloat16>(p, cs, stream);
        case 2: return launch_typed<float, __nv_bfloat16>(p, cs, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace sv
