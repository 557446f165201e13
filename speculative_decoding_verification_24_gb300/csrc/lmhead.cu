// LM head on the 5th-generation tensor cores: logits[M, V] = hidden[M, d] .
// W[d, V] with bf16 inputs and fp32 accumulation, written to an fp32 buffer.
//
// The verify step's target rows are the target model's output head applied
// to the K+1 positions of every sequence ("Speculative decoding",
// denimpatel.github.io interactive course, section "Memory-bound, not
// compute-bound": verification is a forward pass whose query dimension is the
// number of positions, so the head's weights are read once for all of them).
// M = B * (K+1) is small, so the product is computed transposed (swap-AB):
//   D^T[v, m] = sum_k W[k, v] * hidden[m, k]
// with a 128-wide slice of V as the MMA's M dimension (A = W^T, read from the
// V-contiguous W as an MN-major operand) and the M rows of hidden as the MMA's
// N dimension (B = hidden, K-major), N = M rounded up to 16 (at most 256).
//
// Persistent CTAs, one per SM, each taking the 128-column tiles t = block,
// block + grid, ...:
//   warp 0  TMA producer: per LM_BLOCK_K-deep step of d, two 64-column boxes of W and one
//           LM_BLOCK_K x N box of hidden (128-byte / 64-byte swizzle) into an S-stage ring that
//           runs on across tiles; stages complete on mbarriers;
//   warp 1  allocates TMEM (two 128-lane x 256-column accumulators) and one
//           thread issues tcgen05.mma (kind::f16, LM_BLOCK_K / 16 per stage, K = 16 each),
//           committing each stage back to the producer and each finished tile
//           to the epilogue; a tile's MMAs wait until the epilogue has drained
//           the accumulator they reuse;
//   warps 2-3  (sample mode of the verify step) the draft rows' softmax
//           partials over the same tiles, read straight from global memory:
//           they need nothing from the other warps, so they run ahead;
//   warps 4-7  epilogue: tcgen05.ld of the finished accumulator (warp w reads
//           TMEM lanes 32(w-4)...), one coalesced 128-byte store per column and
//           warp, then the accumulator is handed back; it overlaps the next
//           tile's loads and MMAs.
// When the verify step follows (spec_verify_lmhead), the epilogue also
// reduces every row of the tile to one softmax partial (R, s) in the base-2
// domain, or to the row's (max, lowest index) in greedy mode: a warp's 32
// columns are turned over through shared memory so that lane l holds row
// c0 + l, each lane reduces its row over those columns, the four warps'
// partials merge in warp order, and each row's partial merges into the
// CTA's running partial of that row (its tiles in order), written once at the
// end. The verify kernel merges the CTAs' partials instead of streaming the
// target rows again; it re-reads one target row per sequence only for the
// final draw.
// Every mbarrier wait is bounded; a wait that gives up sets SV_FLAG_TIMEOUT,
// the CTA stops issuing work, waits for what it issued and frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <type_traits>

#include "sv_device.cuh"
#include "sv_launch.h"

namespace sv {

constexpr int LM_BLOCK_V = 128;                          // columns of V per tile (MMA M)
// d per stage. 64: one 128-byte row of bf16 per hidden row. (32, the same
// ring bytes in twice as many stages with 64-byte swizzled hidden rows,
// measured 1.6x slower on GB300.)
constexpr int LM_BLOCK_K = 64;
constexpr int LM_A_BYTES = LM_BLOCK_V * LM_BLOCK_K * 2;  // two 64-column boxes of W
constexpr int LM_BOX_BYTES = 64 * LM_BLOCK_K * 2;        // one box of W
constexpr int LM_MAX_STAGES = 12;
// hidden rows are K-major with LM_BLOCK_K * 2 bytes per row: 128-byte (64)
// or 64-byte (32) swizzle; descriptor layout codes 2 and 4
constexpr int LM_B_ROW_BYTES = LM_BLOCK_K * 2;
constexpr uint32_t LM_B_LAYOUT = LM_B_ROW_BYTES == 128 ? 2u : 4u;
static_assert(LM_B_ROW_BYTES == 128 || LM_B_ROW_BYTES == 64, "hidden rows of 64 or 128 bytes");
constexpr int LM_SMEM_BUDGET = 226 * 1024;               // dynamic shared memory (ring + epilogue)
constexpr int LM_THREADS = 256;
constexpr int LM_ACC_COLS = 256;                         // TMEM columns per accumulator
constexpr int LM_TMEM_COLS = 2 * LM_ACC_COLS;
constexpr uint32_t LM_WAIT_LIMIT = 1u << 24;
constexpr int LM_EPI_WARPS = 4;
constexpr int LM_MAX_ROWS = 256;                          // M = B*(K+1) and B*K at most
constexpr int LM_TB_STRIDE = 33;                          // padded row: conflict-free both ways
constexpr int LM_TB_BYTES = LM_EPI_WARPS * 32 * LM_TB_STRIDE * 4;   // per-warp 32 x 32 turn-over
constexpr int LM_WP_BYTES = LM_EPI_WARPS * 256 * 8;                 // per-warp row partials
constexpr int LM_EPI_BYTES = LM_TB_BYTES + LM_WP_BYTES;

struct LmParams {
    int M, d, V, N;     // N: M rounded up to 16
    int stages;         // ring stages (<= LM_MAX_STAGES)
    int tiles;          // ceil(V / LM_BLOCK_V)
    float* out;         // [M, V], or nullptr (partials only: no logit is stored)
    uint32_t* status;   // optional
    float2* parts;      // [grid, M] each CTA's row partials over its tiles, or nullptr (logits only)
    float c;            // log2(e) / temperature (soft partials)
    int part_soft;      // 1: (R, s) softmax partials; 0: (max, lowest index)
    // Sample mode: the draft rows' softmax partials per tile, by warps 2-3.
    const void* draft;  // [Md, V] draft logits (fp32 or bf16), or nullptr
    int Md, draft_f32;  // draft rows; element type
    float2* dparts;     // [grid, Md]
};

// tcgen05 shared-memory matrix descriptor: start address, leading and stride
// byte offsets (all >> 4), descriptor version 1, swizzle layout code
// (2: 128-byte, 4: 64-byte).
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)layout << 61;
    return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B,
// A MN-major, B K-major, N x M shape.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int n, int m) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
          "r"(smem_u32(bar))
        : "memory");
}

// The same load with an L2 eviction policy (W streams through L2 once per
// call: marked evict-first, it does not push out the logits and partials the
// verify step reads next).
__device__ __forceinline__ void tma_load_2d_hint(void* smem_dst, const CUtensorMap* map, int x, int y,
                                                 uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
          "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ bool lm_error(const int* err) { return *(volatile const int*)err != 0; }

// Named barrier 1 over the four epilogue warps (barrier 0 is __syncthreads).
__device__ __forceinline__ void epi_barrier() {
    asm volatile("bar.sync 1, %0;" ::"n"(LM_EPI_WARPS * 32) : "memory");
}

// The same barrier, returning the AND of every epilogue thread's v.
__device__ __forceinline__ bool epi_barrier_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(LM_EPI_WARPS * 32)
        : "memory");
    return r != 0;
}

// Draft-row partials over this CTA's tiles, by one of two warps (w2): lane l
// holds columns v0 + 4l .. v0 + 4l + 3 of a row (V is a multiple of 8, so the
// four are inside the row or past its end together); a warp reduction gives
// the tile's maximum, then R = ceil(max * c) and s = sum 2^(l*c - R) exactly
// as the epilogue forms the target rows' partials. Rows go in batches (32
// bf16 or 16 fp32 rows per warp) whose loads are in flight together: these
// loads compete with the W stream, and only many of them in flight keep the
// two warps ahead of the GEMM. Lane k keeps the running partial of row k of
// each of its batches across the tiles (in tile order) and writes it once,
// at the end: one partial per row and CTA.
// Draft-row loads with an L2 evict-first policy: the verify step needs the
// draft rows again only for one row per sequence, while the fp32 logits this
// kernel writes are what its final draw re-reads; evict-first keeps the 41 MB
// of draft reads (c5) from pushing those logits out of L2.
__device__ __forceinline__ uint4 ld_draft_v4(const void* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ uint2 ld_draft_v2(const void* p, uint64_t pol) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;"
                 : "=r"(v.x), "=r"(v.y)
                 : "l"(p), "l"(pol));
    return v;
}

template <bool F32>
__device__ __forceinline__ void draft_partials(const LmParams& p, int w2, int lane, int my_tiles, const int* err) {
    constexpr int RB = F32 ? 16 : 32;
    constexpr int MAXB = (LM_MAX_ROWS + 2 * RB - 1) / (2 * RB);  // batches per warp
    using Raw = typename std::conditional<F32, uint4, uint2>::type;
    constexpr int ESZ = F32 ? 4 : 2;
    const bool vec = (reinterpret_cast<uintptr_t>(p.draft) & (uintptr_t)(4 * ESZ - 1)) == 0;
    const uint64_t pol = policy_evict_first();
    const float2 empty = pack(SoftPart{-INFINITY, 0.0f});
    float2 run[MAXB];  // indexed at run time: a few bytes of local memory per lane
#pragma unroll
    for (int bi = 0; bi < MAXB; ++bi) run[bi] = empty;
    int li = 0;
    for (; li < my_tiles && !lm_error(err); ++li) {
        const int tile = (int)blockIdx.x + li * (int)gridDim.x;
        const int e = tile * LM_BLOCK_V + 4 * lane;
        const bool in = e < p.V;
#pragma unroll 1
        for (int bi = 0; bi < MAXB; ++bi) {
            const int m0 = w2 * RB + bi * 2 * RB;
            if (m0 >= p.Md) break;
            Raw raw[RB];
#pragma unroll
            for (int k = 0; k < RB; ++k) {
                const bool ok = in && m0 + k < p.Md;
                const char* row = static_cast<const char*>(p.draft) + ((size_t)(m0 + k) * p.V + e) * ESZ;
                if constexpr (F32) {
                    raw[k] = make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
                    if (ok) {
                        if (vec) {
                            raw[k] = ld_draft_v4(row, pol);
                        } else {
                            const uint32_t* r32 = reinterpret_cast<const uint32_t*>(row);
                            raw[k] = make_uint4(__ldg(r32), __ldg(r32 + 1), __ldg(r32 + 2), __ldg(r32 + 3));
                        }
                    }
                } else {
                    raw[k] = make_uint2(0xFF80FF80u, 0xFF80FF80u);  // bf16 -inf pairs
                    if (ok) {
                        if (vec) {
                            raw[k] = ld_draft_v2(row, pol);
                        } else {
                            const unsigned short* r16 = reinterpret_cast<const unsigned short*>(row);
                            raw[k] = make_uint2((uint32_t)__ldg(r16) | ((uint32_t)__ldg(r16 + 1) << 16),
                                                (uint32_t)__ldg(r16 + 2) | ((uint32_t)__ldg(r16 + 3) << 16));
                        }
                    }
                }
            }
            float2 mine = empty;  // lane k: row m0 + k of this batch
#pragma unroll
            for (int k = 0; k < RB; ++k) {
                float x[4];
                if constexpr (F32) {
                    x[0] = __uint_as_float(raw[k].x), x[1] = __uint_as_float(raw[k].y);
                    x[2] = __uint_as_float(raw[k].z), x[3] = __uint_as_float(raw[k].w);
                } else {
                    x[0] = bf16_lo(raw[k].x), x[1] = bf16_hi(raw[k].x), x[2] = bf16_lo(raw[k].y), x[3] = bf16_hi(raw[k].y);
                }
                float mx = max_nan(max_nan(x[0], x[1]), max_nan(x[2], x[3]));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mx = max_nan(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float R = ceilf(mx * p.c);
                const float nR = R == -INFINITY ? 0.0f : -R;
                float s = (ex2(fmaf(x[0], p.c, nR)) + ex2(fmaf(x[1], p.c, nR))) +
                          (ex2(fmaf(x[2], p.c, nR)) + ex2(fmaf(x[3], p.c, nR)));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                if (lane == k) mine = R == -INFINITY ? empty : pack(SoftPart{R, s});
            }
            run[bi] = pack(merge_soft(as_soft(run[bi]), as_soft(mine)));
        }
    }
    // an unfinished CTA (a wait that gave up) reports NaN: its rows are invalid
    const bool done = li == my_tiles;
#pragma unroll
    for (int bi = 0; bi < MAXB; ++bi) {
        const int m = w2 * RB + bi * 2 * RB + lane;
        if (lane < RB && m < p.Md)
            p.dparts[(size_t)blockIdx.x * p.Md + m] = done ? run[bi] : make_float2(__int_as_float(0x7fc00000), 0.0f);
    }
}

__global__ void __launch_bounds__(LM_THREADS, 1)
    lmhead_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_h,
                       LmParams p) {
    extern __shared__ __align__(1024) char smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = p.stages;
    const int b_bytes = p.N * LM_BLOCK_K * 2;
    char* a_ring = smem;                      // S x 16 KB
    char* b_ring = smem + S * LM_A_BYTES;     // S x b_bytes (b_bytes is a multiple of 1 KB)
    float* epi_tb = reinterpret_cast<float*>(b_ring + S * b_bytes);      // LM_TB_BYTES
    float2* epi_wp = reinterpret_cast<float2*>(b_ring + S * b_bytes + LM_TB_BYTES);  // LM_WP_BYTES
    __shared__ __align__(8) uint64_t full[LM_MAX_STAGES], empty[LM_MAX_STAGES];
    __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], mma_done;
    __shared__ uint32_t tmem_base;
    __shared__ int err;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ksteps = p.d / LM_BLOCK_K;
    const int my_tiles = p.tiles > (int)blockIdx.x ? (p.tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 128);  // every epilogue thread
        }
        mbar_init(&mma_done, 1);
        err = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&tmem_base)), "r"(LM_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const uint32_t tmem = tmem_base;
    // A verify launch that follows may start on the SMs this grid leaves free
    // as its CTAs finish; it reads nothing this grid writes before the grid
    // has completed.
    launch_dependents();

    if (warp == 0 && lane == 0) {
        // ---- TMA producer: one continuous ring over all of this CTA's tiles
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_w)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_h)) : "memory");
        const uint64_t w_policy = policy_evict_first();
        int it = 0;
        for (int li = 0; li < my_tiles && !lm_error(&err); ++li) {
            const int v0 = ((int)blockIdx.x + li * (int)gridDim.x) * LM_BLOCK_V;
            // a tile whose second 64 columns lie wholly past V loads only the
            // first box; the MMA rows of the other half are never stored
            const bool second_box = v0 + 64 < p.V;
            const uint32_t stage_tx = (uint32_t)((second_box ? LM_A_BYTES : LM_BOX_BYTES) + b_bytes);
            for (int ks = 0; ks < ksteps; ++ks, ++it) {
                const int s = it % S, n = it / S;
                if (n > 0 && !mbar_wait(&empty[s], (n - 1) & 1, LM_WAIT_LIMIT)) {
                    atomicExch(&err, 1);
                    break;
                }
                mbar_arrive_expect_tx(&full[s], stage_tx);
                char* a = a_ring + s * LM_A_BYTES;
                tma_load_2d_hint(a, &tm_w, v0, ks * LM_BLOCK_K, &full[s], w_policy);
                if (second_box) tma_load_2d_hint(a + LM_BOX_BYTES, &tm_w, v0 + 64, ks * LM_BLOCK_K, &full[s], w_policy);
                tma_load_2d(b_ring + s * b_bytes, &tm_h, ks * LM_BLOCK_K, 0, &full[s]);
            }
        }
        // every load issued has landed before this thread leaves: the last
        // min(S, it) loads are the latest phase of their stages
        for (int q = it - S > 0 ? it - S : 0; q < it; ++q)
            (void)mbar_wait(&full[q % S], (q / S) & 1, LM_WAIT_LIMIT);
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        const uint32_t idesc = umma_idesc_bf16(p.N, LM_BLOCK_V);
        int it = 0;
        bool ok = true;
        for (int li = 0; li < my_tiles && ok; ++li) {
            const int a = li & 1;
            if (li >= 2 && !mbar_wait(&acc_empty[a], ((li >> 1) - 1) & 1, LM_WAIT_LIMIT)) {
                ok = false;
                break;
            }
            tmem_fence_after();
            const uint32_t acc = tmem + (uint32_t)(a * LM_ACC_COLS);
            for (int ks = 0; ks < ksteps; ++ks, ++it) {
                const int s = it % S, n = it / S;
                if (!mbar_wait(&full[s], n & 1, LM_WAIT_LIMIT)) {
                    ok = false;
                    break;
                }
                tmem_fence_after();
                const uint32_t a0 = smem_u32(a_ring + s * LM_A_BYTES);
                const uint32_t b0 = smem_u32(b_ring + s * b_bytes);
#pragma unroll
                for (int kk = 0; kk < LM_BLOCK_K / 16; ++kk) {
                    // A (MN-major, 128-byte swizzle): 16 rows of d = two 8-row
                    //   swizzle atoms (2 KB); LBO = the second 64-wide block of V
                    //   (the second box), SBO = 8 rows.
                    // B (K-major): 16 elements of d = 32 bytes inside the row;
                    //   SBO = 8 rows of the swizzle atom.
                    const uint64_t ad = umma_desc(a0 + kk * 2048, LM_BOX_BYTES, 1024, 2u);
                    const uint64_t bd = umma_desc(b0 + kk * 32, 16, 8 * LM_B_ROW_BYTES, LM_B_LAYOUT);
                    umma_bf16(acc, ad, bd, idesc, (ks | kk) != 0);
                }
                umma_commit(&empty[s]);  // the stage is free once these MMAs completed
            }
            if (!ok) break;
            umma_commit(&acc_full[a]);  // the tile's accumulator is complete
        }
        if (!ok) atomicExch(&err, 1);
        // every MMA issued has completed before TMEM is released
        umma_commit(&mma_done);
        (void)mbar_wait(&mma_done, 0, LM_WAIT_LIMIT);
    } else if ((warp == 2 || warp == 3) && p.dparts) {
        // ---- draft rows: every row's partial over each of this CTA's tiles
        if (p.draft_f32) draft_partials<true>(p, warp - 2, lane, my_tiles, &err);
        else draft_partials<false>(p, warp - 2, lane, my_tiles, &err);
    } else if (warp >= 4) {
        // ---- epilogue: TMEM -> registers -> global (coalesced per column)
        const int q = warp - 4;
        float* tb = epi_tb + q * 32 * LM_TB_STRIDE;
        // thread t's running partials of rows t and t + 128 over this CTA's
        // tiles (merged in tile order; written once, at the end)
        const float2 empty = p.part_soft ? pack(SoftPart{-INFINITY, 0.0f}) : pack(ArgPart{-INFINITY, INT_MAX});
        float2 run0 = empty, run1 = empty;
        int li = 0;
        for (; li < my_tiles; ++li) {
            const int a = li & 1;
            bool ok = mbar_wait(&acc_full[a], (li >> 1) & 1, LM_WAIT_LIMIT);
            tmem_fence_after();
            if (!ok) atomicExch(&err, 1);
            // One decision for all four warps (tcgen05.ld is warp-collective,
            // and the warps meet at the partial merge below). This barrier
            // also keeps a warp from writing the next tile's partials before
            // every warp has merged this tile's.
            ok = epi_barrier_and(ok && !lm_error(&err));
            if (!ok) break;
            const int tile = (int)blockIdx.x + li * (int)gridDim.x;
            const int vw = tile * LM_BLOCK_V + 32 * q;  // this warp's first column
            const int v = vw + lane;
            const int nv = p.V - vw;                     // valid columns of the warp (may be <= 0)
            const uint32_t acc = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(a * LM_ACC_COLS);
            for (int c0 = 0; c0 < p.N; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(acc + (uint32_t)c0, r);
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int m = c0 + c;
                    if (p.out && m < p.M && v < p.V) p.out[(size_t)m * p.V + v] = __uint_as_float(r[c]);
                }
                if (p.parts) {
                    // turn the 32 x 32 block over: lane l then holds row c0 + l
                    // at the warp's 32 columns, in column order
#pragma unroll
                    for (int c = 0; c < 32; ++c) tb[c * LM_TB_STRIDE + lane] = __uint_as_float(r[c]);
                    __syncwarp();
                    float x[32];
#pragma unroll
                    for (int k = 0; k < 32; ++k) x[k] = tb[lane * LM_TB_STRIDE + k];
                    __syncwarp();  // the next block overwrites tb
                    float2 part;
                    if (p.part_soft) {
                        float mx = -INFINITY;
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            if (k < nv) mx = max_nan(mx, x[k]);
                        const float R = ceilf(mx * p.c);  // -inf, +inf and NaN pass through
                        const float nR = R == -INFINITY ? 0.0f : -R;
                        float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
                        for (int k = 0; k < 32; k += 2) {
                            if (k < nv) s0 += ex2(fmaf(x[k], p.c, nR));
                            if (k + 1 < nv) s1 += ex2(fmaf(x[k + 1], p.c, nR));
                        }
                        part = R == -INFINITY ? pack(SoftPart{-INFINITY, 0.0f}) : pack(SoftPart{R, s0 + s1});
                    } else {
                        // the first maximum in column order; a NaN replaces any number
                        ArgPart best{-INFINITY, INT_MAX};
#pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            const bool take = k < nv && (x[k] > best.v || (is_nan(x[k]) && !is_nan(best.v)));
                            if (take) best = ArgPart{x[k], vw + k};
                        }
                        part = pack(best);
                    }
                    epi_wp[q * 256 + c0 + lane] = part;  // c0 + lane < N <= 256
                }
            }
            tmem_fence_before();
            mbar_arrive(&acc_empty[a]);
            if (p.parts) {
                // the four warps' partials of every row, merged in warp order
                epi_barrier();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int m = (int)threadIdx.x - 128 + h * 128;
                    if (m < p.M) {
                        float2 acc2 = epi_wp[m];
#pragma unroll
                        for (int w = 1; w < LM_EPI_WARPS; ++w)
                            acc2 = p.part_soft ? pack(merge_soft(as_soft(acc2), as_soft(epi_wp[w * 256 + m])))
                                               : pack(merge_arg(as_arg(acc2), as_arg(epi_wp[w * 256 + m])));
                        float2& run = h == 0 ? run0 : run1;
                        run = p.part_soft ? pack(merge_soft(as_soft(run), as_soft(acc2)))
                                          : pack(merge_arg(as_arg(run), as_arg(acc2)));
                    }
                }
            }
        }
        if (p.parts) {
            // one partial per row and CTA; an unfinished CTA (a wait that
            // gave up) reports NaN, so the verify marks its rows invalid
            const bool done = li == my_tiles;
            const float2 nan2 = make_float2(__int_as_float(0x7fc00000), 0.0f);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int m = (int)threadIdx.x - 128 + h * 128;
                if (m < p.M) p.parts[(size_t)blockIdx.x * p.M + m] = done ? (h == 0 ? run0 : run1) : nan2;
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tmem_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(LM_TMEM_COLS)
                     : "memory");
    }
    if (threadIdx.x == 0 && err && p.status) atomicOr(p.status, (unsigned)SV_FLAG_TIMEOUT);
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static std::atomic<void*> fn{nullptr};
    void* f = fn.load(std::memory_order_acquire);
    if (!f) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn.store(f, std::memory_order_release);
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

// 2-D bf16 tensor map over a row-major [rows, cols] matrix, box [box_rows,
// box_cols] with box_cols * 2 bytes inner (128: 128-byte swizzle, 64: 64-byte
// swizzle), zero fill out of bounds.
static bool encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                           uint32_t box_rows, uint32_t box_cols) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode();
    if (!encode) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw = box_cols * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Ring stages that fit beside the epilogue's buffers (needed only when the
// epilogue writes partials).
static int lmhead_stages(int N, bool parts) {
    const int stage = LM_A_BYTES + N * LM_BLOCK_K * 2;
    const int st = (LM_SMEM_BUDGET - 1024 - (parts ? LM_EPI_BYTES : 0)) / stage;
    return st < LM_MAX_STAGES ? st : LM_MAX_STAGES;
}

static std::atomic<int> g_lm_sms[64];

cudaError_t launch_lmhead_gemm(const void* hidden, const void* W, int M, int d, int V, float* out,
                               float2* parts, float c, int part_soft, const LmDraftParts* dp,
                               uint32_t* status, cudaStream_t stream, int* grid_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    static std::atomic<int> attr_done[64];
    if (!attr_done[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(lmhead_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, LM_SMEM_BUDGET);
        if (e != cudaSuccess) return e;
        attr_done[dev].store(1, std::memory_order_release);
    }
    int sms = g_lm_sms[dev].load(std::memory_order_acquire);
    if (sms == 0) {
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_lm_sms[dev].store(sms, std::memory_order_release);
    }
    LmParams p;
    p.M = M;
    p.d = d;
    p.V = V;
    p.N = (M + 15) / 16 * 16;
    p.stages = lmhead_stages(p.N, parts != nullptr);
    p.tiles = (V + LM_BLOCK_V - 1) / LM_BLOCK_V;
    p.out = out;
    p.status = status;
    p.parts = parts;
    p.c = c;
    p.part_soft = part_soft;
    p.draft = dp ? dp->draft : nullptr;
    p.Md = dp ? dp->Md : 0;
    p.draft_f32 = dp ? dp->draft_f32 : 0;
    p.dparts = dp ? dp->dparts : nullptr;
    CUtensorMap tm_w, tm_h;
    if (!encode_bf16_2d(&tm_w, W, (uint64_t)d, (uint64_t)V, LM_BLOCK_K, 64) ||
        !encode_bf16_2d(&tm_h, hidden, (uint64_t)M, (uint64_t)d, (uint32_t)p.N, LM_BLOCK_K))
        return cudaErrorInvalidValue;
    const int smem = 1024 + p.stages * (LM_A_BYTES + p.N * LM_BLOCK_K * 2) + (parts ? LM_EPI_BYTES : 0);
    const dim3 grid((unsigned)(p.tiles < sms ? p.tiles : sms));
    if (grid_out) *grid_out = (int)grid.x;
    lmhead_gemm_kernel<<<grid, LM_THREADS, smem, stream>>>(tm_w, tm_h, p);
    return cudaGetLastError();
}

}  // namespace sv
