// Prompt lookup drafting on the GPU ("Inference-4" (brunomaga.github.io),
// section "Prompt lookup decoding"): the drafts are the tokens that followed
// the most recent earlier occurrence of the sequence's last n-gram, trying
// n = max_ngram first; none when no n-gram of length 1..max_ngram recurs.
//
// A window that ends at position e (e <= L-2, so it ends before the last
// token) matches the last n tokens for every n up to ml(e), the length of the
// common suffix of seq[..e] and seq[..L-1] (capped at max_ngram). The n that
// wins is the largest ml over all e, and its most recent window has the
// largest e among those: so one max-reduction of the key (ml(e), e) over all
// positions gives both. The drafts are then seq[e+1 .. e+n_drafts], cut at L.
//
// One cluster per sequence: CTA r of the cluster scans the r-th contiguous
// part of the positions, the CTAs' keys meet in rank 0's shared memory, and
// rank 0 writes the drafts.
#include <cooperative_groups.h>

#include <atomic>
#include <cstdint>

#include "sv_device.cuh"
#include "sv_launch.h"

namespace cg = cooperative_groups;

namespace sv {

constexpr int PL_THREADS = 256;
constexpr int PL_PER = 16;                        // tokens per thread and tile
constexpr int PL_TILE = PL_THREADS * PL_PER;      // 4096 tokens per tile
constexpr int PL_HALO = PL_MAX_NGRAM;             // tokens before a tile a window may reach
constexpr int PL_MAX_CLUSTER = 8;

// A CTA's part streams through shared memory a tile at a time: every thread
// issues its PL_PER coalesced loads of the next tile (and the tile's halo of
// PL_HALO earlier tokens) before the CTA scans the current one, so one load
// latency covers a whole tile.
__global__ void __launch_bounds__(PL_THREADS) prompt_lookup_kernel(const int32_t* tokens, const int32_t* lengths,
                                                                   int L_max, int max_ngram, int n_drafts,
                                                                   int32_t* out_drafts, int32_t* out_n) {
    __shared__ int32_t suffix[PL_MAX_NGRAM];
    __shared__ int32_t tile[2][PL_HALO + PL_TILE];
    __shared__ long long warp_best[PL_THREADS / 32];
    __shared__ long long cta_best[PL_MAX_CLUSTER];  // rank 0: every CTA's key
    __shared__ int32_t cta_drafts[PL_MAX_CLUSTER][PL_MAX_DRAFTS];  // rank 0: the drafts after each key
    cg::cluster_group cluster = cg::this_cluster();
    const int CS = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int b = (int)blockIdx.x / CS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t* seq = tokens + (size_t)b * L_max;
    int32_t* out = out_drafts + (size_t)b * n_drafts;
    // The parts are cut from the window ends the buffer allows (0 .. L_max-2),
    // not the sequence's own, so that the first tile's loads go out before
    // the length has arrived; the scan then stops at the sequence's last
    // window end, L-2. (Loads past the sequence stay inside its row of the
    // buffer and are never compared.)
    const int n_buf = L_max - 1 > 0 ? L_max - 1 : 0;
    const int per = (n_buf + CS - 1) / CS;
    const int p0 = min(n_buf, rank * per), p1_buf = min(n_buf, p0 + per);
    int32_t r[PL_PER], h = 0;
    auto load = [&](int t0, int lim) {
#pragma unroll
        for (int k = 0; k < PL_PER; ++k) {
            const int i = t0 + k * PL_THREADS + tid;
            r[k] = i < lim ? __ldg(seq + i) : 0;
        }
        if (tid < PL_HALO) {
            const int i = t0 - PL_HALO + tid;
            h = i >= 0 ? __ldg(seq + i) : 0;
        }
    };
    auto store = [&](int buf) {
#pragma unroll
        for (int k = 0; k < PL_PER; ++k) tile[buf][PL_HALO + k * PL_THREADS + tid] = r[k];
        if (tid < PL_HALO) tile[buf][tid] = h;
    };
    if (p0 < p1_buf) load(p0, p1_buf);  // in flight while the length arrives
    const int L = __ldg(lengths + b);
    const bool valid = L >= 0 && L <= L_max;
    if (valid && tid < max_ngram && tid < L) suffix[tid] = __ldg(seq + (L - 1 - tid));
    if (!valid) {  // the same for every CTA of the cluster: none takes part in a cluster barrier
        if (rank == 0) {
            for (int i = tid; i < n_drafts; i += PL_THREADS) out[i] = -1;
            if (tid == 0) out_n[b] = -1;
        }
        return;
    }
    // Every CTA of the cluster has started once this phase of the cluster
    // barrier completes; its wait comes just before rank 0's shared memory is
    // written, by which time it has long completed.
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    // windows end at e = 0 .. L-2; this CTA takes e in [p0, p1)
    const int n_pos = L - 1 > 0 ? L - 1 : 0;
    const int p1 = max(p0, min(p1_buf, n_pos));
    const int n_tiles = (p1 - p0 + PL_TILE - 1) / PL_TILE;
    // (ml << 32) | e, the largest over this thread's windows. A window whose
    // last token differs from the sequence's last has ml = 0, and the largest
    // such key is this CTA's last window end, p1 - 1: so only windows that
    // match the last token need the rest of the comparison.
    long long best = (tid == 0 && p1 > p0) ? (long long)(p1 - 1) : -1;
    if (n_tiles > 0) store(0);
    __syncthreads();
    const int32_t s0 = n_tiles > 0 ? suffix[0] : 0;
    for (int ti = 0; ti < n_tiles; ++ti) {
        const int t0 = p0 + ti * PL_TILE, buf = ti & 1;
        if (ti + 1 < n_tiles) load(t0 + PL_TILE, p1);  // in flight during the scan below
        const int32_t* tl = tile[buf] + PL_HALO - t0;  // tl[i] = token i for t0 - PL_HALO <= i < t0 + PL_TILE
        // this thread's positions of the tile read at once, then compared
        int32_t v[PL_PER];
#pragma unroll
        for (int k = 0; k < PL_PER; ++k) {
            const int e = t0 + k * PL_THREADS + tid;
            v[k] = e < p1 ? tl[e] : 0;
        }
#pragma unroll
        for (int k = 0; k < PL_PER; ++k) {
            const int e = t0 + k * PL_THREADS + tid;
            if (e < p1 && v[k] == s0) {
                int ml = 1;
                while (ml < max_ngram && e - ml >= 0 && tl[e - ml] == suffix[ml]) ++ml;
                const long long key = ((long long)ml << 32) | (unsigned)e;
                best = key > best ? key : best;
            }
        }
        if (ti + 1 < n_tiles) store(buf ^ 1);  // nobody reads that buffer in this round
        __syncthreads();
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const long long other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        best = other > best ? other : best;
    }
    if (lane == 0) warp_best[warp] = best;
    __syncthreads();
    // Each CTA reads the drafts that follow its own best window before the
    // cluster exchange (the reads overlap the barrier), and hands them to
    // rank 0 with its key: rank 0 then only picks, with no dependent load
    // after the exchange.
    int32_t dr[PL_MAX_DRAFTS / 32];
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
#pragma unroll
        for (int k = 0; k < PL_MAX_DRAFTS / 32; ++k) {
            const int i = k * 32 + lane;
            dr[k] = i < avail ? __ldg(seq + (e + 1 + i)) : -1;
        }
    }
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // every CTA has started
    if (warp == 0) {
        int32_t* dst = cluster.map_shared_rank(&cta_drafts[0][0], 0) + rank * PL_MAX_DRAFTS;
#pragma unroll
        for (int k = 0; k < PL_MAX_DRAFTS / 32; ++k)
            if (k * 32 + lane < n_drafts) dst[k * 32 + lane] = dr[k];
        if (lane == 0) cluster.map_shared_rank(cta_best, 0)[rank] = best;
    }
    cluster.sync();
    if (rank == 0 && warp == 0) {
        best = lane < CS ? cta_best[lane] : -1;
        int from = lane < CS ? lane : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const long long other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
            const int other_from = __shfl_xor_sync(0xFFFFFFFFu, from, o);
            if (other > best) {
                best = other;
                from = other_from;
            }
        }
        // keys are distinct across CTAs (different window ends), except -1
        // for a CTA without windows, which never wins over a real key
        const int ml = best < 0 ? 0 : (int)(best >> 32);
        const int e = best < 0 ? -1 : (int)(best & 0xFFFFFFFFLL);
        const int avail = ml > 0 ? min(n_drafts, L - 1 - e) : 0;
        for (int i = lane; i < n_drafts; i += 32) out[i] = i < avail ? cta_drafts[from][i] : -1;
        if (lane == 0) out_n[b] = avail;
    }
}

// ---------------------------------------------------------------------------
// Whole-context variant, for contexts of at most PLW_MAX_L tokens: one CTA
// per sequence holds its entire context in shared memory. Tile 0 is copied
// before the length has arrived, the other tiles holding positions < L right
// after; the last tokens (the n-gram to match) are read directly at the same
// time. The scan then reads shared memory only, and so do the drafts: no
// cluster exchange, and no dependent global load after the scan.
// ---------------------------------------------------------------------------
constexpr int PLW_TILE = 4096;     // tokens per bulk copy (16 KB)
constexpr int PLW_MAX_TILES = 6;
constexpr int PLW_MAX_L = PLW_TILE * PLW_MAX_TILES;  // 24576 tokens, 96 KB of shared memory
constexpr uint32_t PLW_WAIT_LIMIT = 1u << 22;        // polls before a copy's wait gives up
constexpr int PLW_SPREAD_BYTES = 80 * 1024;        // more than a third of an SM's shared memory

__global__ void __launch_bounds__(PL_THREADS) prompt_lookup_whole_kernel(const int32_t* tokens, const int32_t* lengths,
                                                                         int L_max, int max_ngram, int n_drafts,
                                                                         int32_t* out_drafts, int32_t* out_n) {
    extern __shared__ __align__(128) int32_t ctx[];  // ctx[i] = token i of the sequence
    __shared__ uint64_t bar[PLW_MAX_TILES];
    __shared__ int32_t suffix[PL_MAX_NGRAM];
    __shared__ long long warp_best[PL_THREADS / 32];
    __shared__ int s_err;
    const int b = (int)blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t* seq = tokens + (size_t)b * L_max;
    int32_t* out = out_drafts + (size_t)b * n_drafts;
    // L_max is a multiple of 4 and the rows are 16-byte aligned (checked on
    // the host), so every copy below is a whole number of 16-byte units
    // inside the sequence's row.
    const int n0 = min(PLW_TILE, L_max);
    // The next call may launch now; this one reads its inputs only once the
    // work ahead of it has completed (the commit step writes the contexts).
    launch_dependents();
    if (tid == 0) {
        for (int t = 0; t < PLW_MAX_TILES; ++t) mbar_init(&bar[t], 1);
        s_err = 0;
        fence_barrier_init();
    }
    grid_dependency_wait();
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar[0], (uint32_t)n0 * 4u);
        bulk_g2s(ctx, seq, (uint32_t)n0 * 4u, &bar[0]);
    }
    const int L = __ldg(lengths + b);
    const bool valid = L >= 0 && L <= L_max;
    const int nt = valid ? (L + PLW_TILE - 1) / PLW_TILE : 0;  // tiles holding positions < L
    const int Lc = valid ? min((L + 3) & ~3, L_max) : 0;     // tokens copied, whole 16-byte units
    if (tid == 0) {
        for (int t = 1; t < nt; ++t) {
            const int n = min(PLW_TILE, Lc - t * PLW_TILE);
            mbar_arrive_expect_tx(&bar[t], (uint32_t)n * 4u);
            bulk_g2s(ctx + t * PLW_TILE, seq + t * PLW_TILE, (uint32_t)n * 4u, &bar[t]);
        }
    }
    if (valid && tid < max_ngram && tid < L) suffix[tid] = __ldg(seq + (L - 1 - tid));
    __syncthreads();
    // Window ends e = 0 .. L-2 (see prompt_lookup_kernel): key (ml << 32) | e.
    // Only windows whose last token equals the sequence's last need the rest
    // of the comparison; the others have ml = 0 and never yield drafts.
    long long best = -1;
    const int n_pos = L - 1 > 0 ? L - 1 : 0;
    const int32_t s0 = (valid && L > 0) ? suffix[0] : 0;
    for (int t = 0; t < nt; ++t) {
        if (!mbar_wait(&bar[t], 0, PLW_WAIT_LIMIT)) {
            atomicExch(&s_err, 1);
            break;
        }
        // This thread's positions of the tile are read first, all at once (one
        // shared-memory latency per tile rather than one per position), then
        // compared. Measured on GB300, 256 contexts of up to 16384 tokens,
        // calls back to back: 6.4 us per call reading and comparing one
        // position at a time, 5.1 us reading them at once, 4.9 us with at most
        // two CTAs per SM (see the launch).
        constexpr int PER_T = PLW_TILE / PL_THREADS;
        int32_t v[PER_T];
#pragma unroll
        for (int k = 0; k < PER_T; ++k) {
            const int e = t * PLW_TILE + k * PL_THREADS + tid;
            v[k] = e < n_pos ? ctx[e] : 0;
        }
#pragma unroll
        for (int k = 0; k < PER_T; ++k) {
            const int e = t * PLW_TILE + k * PL_THREADS + tid;
            if (e < n_pos && v[k] == s0) {
                int ml = 1;
                while (ml < max_ngram && e - ml >= 0 && ctx[e - ml] == suffix[ml]) ++ml;
                const long long key = ((long long)ml << 32) | (unsigned)e;
                best = key > best ? key : best;
            }
        }
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
        const bool ok = valid && !s_err;
        const int ml = (best < 0 || !ok) ? 0 : (int)(best >> 32);
        const int e = best < 0 ? -1 : (int)(best & 0xFFFFFFFFLL);
        // drafts: ctx[e+1 .. e+n_drafts], cut at the end of the sequence
        // (every position below L is in shared memory)
        const int avail = ml > 0 ? min(n_drafts, L - 1 - e) : 0;
        for (int i = lane; i < n_drafts; i += 32) out[i] = i < avail ? ctx[e + 1 + i] : -1;
        if (lane == 0) out_n[b] = ok ? avail : -1;
    }
    // every copy this CTA issued has landed before it exits (bounded)
    if (tid == 0) {
        (void)mbar_wait(&bar[0], 0, PLW_WAIT_LIMIT);
        for (int t = 1; t < nt; ++t) (void)mbar_wait(&bar[t], 0, PLW_WAIT_LIMIT);
    }
}

// CTAs of the lookup kernel that fit on the GPU at once (per device, cached).
static std::atomic<int> g_pl_resident[64];

static int pl_resident_ctas() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int n = g_pl_resident[dev].load(std::memory_order_acquire);
    if (n == 0) {
        int per_sm = 0, sms = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, prompt_lookup_kernel, PL_THREADS, 0) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        n = per_sm * sms;
        g_pl_resident[dev].store(n, std::memory_order_release);
    }
    return n;
}

// The cluster size: one CTA per tile of the longest possible context, at most
// PL_MAX_CLUSTER, and no more than keeps the whole grid resident at once (a
// CTA then scans several tiles, the next one's loads in flight during the
// scan of the current one).
static std::atomic<int> g_plw_attr[64];

cudaError_t launch_prompt_lookup(const int32_t* tokens, const int32_t* lengths, int B, int L_max,
                                 int max_ngram, int n_drafts, int32_t* out_drafts, int32_t* out_n,
                                 cudaStream_t stream) {
    if (L_max <= PLW_MAX_L && L_max % 4 == 0 && (reinterpret_cast<uintptr_t>(tokens) & 15u) == 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64 || !g_plw_attr[dev].load(std::memory_order_acquire)) {
            e = cudaFuncSetAttribute(prompt_lookup_whole_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     PLW_MAX_L * 4);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) g_plw_attr[dev].store(1, std::memory_order_release);
        }
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        cfg.gridDim = dim3((unsigned)B, 1, 1);
        cfg.blockDim = dim3(PL_THREADS, 1, 1);
        // At least PLW_SPREAD_BYTES, so that no SM holds more than two CTAs:
        // with three on some SMs and one on others, the SMs with three set the
        // call's time.
        cfg.dynamicSmemBytes = (size_t)(L_max * 4 > PLW_SPREAD_BYTES ? L_max * 4 : PLW_SPREAD_BYTES);
        cfg.stream = stream;
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, prompt_lookup_whole_kernel, tokens, lengths, L_max, max_ngram, n_drafts,
                                  out_drafts, out_n);
    }
    int cs = (L_max + PL_TILE - 1) / PL_TILE;
    cs = cs < 1 ? 1 : cs > PL_MAX_CLUSTER ? PL_MAX_CLUSTER : cs;
    while (cs & (cs - 1)) ++cs;  // a power of two (1, 2, 4, 8)
    const int resident = pl_resident_ctas();
    while (cs > 1 && resident > 0 && (long long)B * cs > resident) cs >>= 1;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)(B * cs), 1, 1);
    cfg.blockDim = dim3(PL_THREADS, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prompt_lookup_kernel, tokens, lengths, L_max, max_ngram, n_drafts,
                              out_drafts, out_n);
}

}  // namespace sv

namespace sv {

// Commit step of a decode loop: sequence b appends its n_accepted[b] accepted
// drafts and the token after them (out_tokens[b, 0..n]) to its context and
// advances its length, up to L_max. One warp per sequence (K + 1 <= 32).
__global__ void commit_kernel(int32_t* tokens, int32_t* lengths, int B, int L_max, const int32_t* out_tokens,
                              const int32_t* n_accepted, int K, int32_t* out_n_committed) {
    // launched early: the next call may launch now, and this one reads the
    // verify step's outputs only once the work ahead of it has completed
    launch_dependents();
    grid_dependency_wait();
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
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)((B + WARPS - 1) / WARPS), 1, 1);
    cfg.blockDim = dim3(WARPS * 32, 1, 1);
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, commit_kernel, tokens, lengths, B, L_max, out_tokens, n_accepted, K,
                              out_n_committed);
}

}  // namespace sv
