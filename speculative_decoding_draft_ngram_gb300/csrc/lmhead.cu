// Fused LM head + verify statistics on the fifth-generation tensor cores.
//
// The last step of the target model's forward, logits = h W^T (h: the K + 1
// hidden states of every sequence, W: the [V, d] LM head), computed tile by
// tile with tcgen05.mma, and in the same kernel's epilogue the per-block
// quantities that the verify pass would otherwise stream the logits for: for
// every row and every 256-id noise block, the block's largest logit and the
// block's softmax record (largest transformed value m and the sum of
// exp((z - m) / T)).  The decision kernel then runs on these records, and it
// reads the logits back only where a decision needs a single value (the
// draft's logit, the blocks that can hold the sampled token, a tie).
//
// Follows the pages' description of the verify step (SwiftLM page, the
// Leviathan paragraph: the target's logits of the K + 1 positions decide the
// drafts) and of the engine's tensor path (AX Engine page, "Core Technical
// Architecture & Methods": the forward's operations run as GPU tensor ops).
//
// Layout of the work: one CTA per SM, persistent; tiles of 128 rows x 256
// vocab ids (one noise block).  When the row tiles pair up, CTAs run in
// clusters of two: the two take the row tiles of a pair for the same vocab
// tile, and each loads half of that W tile and multicasts it to both, so
// each SM reads a third less from L2 than a lone CTA would (an odd number of
// row tiles runs single CTAs, each loading its whole W tile).  Work is
// ordered row tiles first, so the CTAs running at the same time share their
// W tiles through L2.
// Warp 0 issues the TMA loads (128-byte swizzled, 64 hidden elements per
// stage, a 4-stage ring), warp 1 owns the tensor memory (two 256-column
// accumulators) and one of its threads issues the MMAs, warps 2-5 read an
// accumulator back (tcgen05.ld), round it to bf16 (the logits' dtype), store
// it and reduce it while the next tile's MMAs run.  A ring stage is refilled
// once the MMAs of both CTAs have read it (each CTA's MMA completion arrives
// on both CTAs' barriers).
#include <cuda.h>

#include "verify.cuh"

namespace specng {

constexpr int kHM = 128;        // rows of a tile (tensor-memory lanes)
constexpr int kHN = 256;        // vocab ids of a tile: one noise block
constexpr int kHK = 64;         // hidden elements per stage: 128 bytes of bf16, one swizzle span
constexpr int kHStages = 4;
constexpr int kHThreads = 192;  // warp 0 TMA, warp 1 tensor memory + MMA, warps 2-5 epilogue
constexpr uint32_t kHABytes = kHM * kHK * 2;  // 16 KB
constexpr uint32_t kHBBytes = kHN * kHK * 2;  // 32 KB
constexpr uint32_t kHTmemCols = 2 * kHN;      // two accumulators
static_assert(kHN == (1 << kNoiseBlockShift), "a tile's vocab range is one noise block");
constexpr size_t kHSmem = kHStages * (kHABytes + kHBBytes) + 1024;  // + alignment slack
// CTAs of a cluster (CL, a template parameter): 2 (each loads half of the W tile
// for both) when the row tiles pair up, else 1 (a lone CTA loads its whole W tile).

struct LmHeadArgs {
    CUtensorMap tmA;  // hidden [rows, d] bf16: box {64, 128}, 128-byte swizzle
    CUtensorMap tmB;  // weight [V, d] bf16: box {64, 128} (half a tile), 128-byte swizzle
    CUtensorMap tmC;  // logits [rows, V] bf16: box {32, 32}, no swizzle (the epilogue's stores)
    int rows, d, ntm, ntn;
    __nv_bfloat16* logits;  // [rows, V]
    VerifyDev P;
};

// ---- tcgen05 / TMA helpers (sm_100 family PTX)

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major bf16 tile written by TMA with
// the 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart
// (stride byte offset), the leading byte offset unused, version 1.
__device__ __forceinline__ uint64_t sdesc_k128(uint32_t saddr) {
    uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor of kind::f16: bf16 A and B (K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t dtmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dtmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}
// the mbarrier completes once every MMA issued so far by this thread is done
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 consecutive fp32 columns of the warp's 32 lanes: lane i gets row i.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Loaded once and written to the same offset in every CTA of `mask`, each of
// whose barrier at bar's offset receives the bytes.
__device__ __forceinline__ void tma_load_2d_mc(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* bar,
                                               uint16_t mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster [%0], [%1, {%2, "
        "%3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar)), "h"(mask)
        : "memory");
}
// The barrier at bar's offset in every CTA of `mask` gets one arrival once the
// MMAs issued so far by this thread are done.
__device__ __forceinline__ void tc_commit_mc(uint64_t* bar, uint16_t mask) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "h"(mask)
                 : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared -> global tile store; the part of the box outside the tensor is not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, int x, int y, const void* src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(tm)),
                 "r"(x), "r"(y), "r"(smem_u32(src))
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// The source of all but the last n committed stores has been read.
template <int N>
__device__ __forceinline__ void tma_store_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// A fp32 accumulator rounded to the logits' dtype (round to nearest even), as bits and as a value.
__device__ __forceinline__ uint32_t bf16_bits(float f) { return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(f))); }

template <int CL, bool GREEDY, bool SOFTCAP>
__global__ void __launch_bounds__(kHThreads, 1) lmhead_verify_kernel(const __grid_constant__ LmHeadArgs A) {
    static_assert(CL == 1 || CL == 2, "clusters of one or two CTAs");
    constexpr uint32_t kBPart = kHBBytes / CL;    // the W rows one CTA loads (for every CTA of the cluster)
    constexpr uint16_t kMask = (1u << CL) - 1u;   // every CTA of the cluster
    extern __shared__ uint8_t s_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(s_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + kHStages * kHABytes;
    __shared__ __align__(8) uint64_t s_full[kHStages], s_empty[kHStages], s_accf[2], s_acce[2], s_done;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    // epilogue staging: per warp two boxes of 32 rows x 32 bf16 columns, row-major,
    // written by the warp and stored by TMA while the next one fills
    __shared__ __align__(128) uint4 s_ep[4][2][32 * 4];
    const VerifyDev& P = A.P;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kHStages; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], CL);  // the MMA completions of every CTA of the cluster
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_accf[i], 1);
            mbar_init(&s_acce[i], 4);
        }
        mbar_init(&s_done, 1);
        s_abort = 0;
        mbar_init_fence();
    }
    if (warp == 1) tmem_alloc(&s_tmem, kHTmemCols);
    // the hidden states may come from the kernel before this one, and the records and
    // logits written here may still be read by the previous call's decision kernel
    pdl_wait();
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the other CTA's barriers are initialised before anything is multicast to them
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const int rank = static_cast<int>(cluster_rank());
    const int cid = blockIdx.x / CL, ncl = gridDim.x / CL;
    const int npm = (A.ntm + CL - 1) / CL;  // row-tile groups (pairs, or single tiles)
    const int npairs = npm * A.ntn;  // work units: a row-tile group and a vocab tile
    const int nk = A.d / kHK;
    volatile int* abort_flag = &s_abort;
    auto give_up = [&]() {
        raise_status(P.status, SPECNG_DEV_TIMEOUT);
        *abort_flag = 1;
    };

    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            int st = 0, it = 0;
            for (int pr = cid; pr < npairs && !*abort_flag; pr += ncl) {
                const int tm = CL * (pr % npm) + rank, tn = pr / npm;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    if (it >= kHStages && !mbar_wait_bounded(&s_empty[st], ((it / kHStages) + 1) & 1)) {
                        give_up();
                        break;
                    }
                    // this stage's bytes: my A tile and the W tile (in a cluster of two, my half
                    // of it and the other CTA's half, each multicast to both)
                    mbar_add_tx(&s_full[st], kHABytes + kHBBytes);
                    tma_load_2d(sA + st * kHABytes, &A.tmA, kb * kHK, tm * kHM, &s_full[st]);
                    if constexpr (CL == 1)
                        tma_load_2d(sB + st * kHBBytes, &A.tmB, kb * kHK, tn * kHN, &s_full[st]);
                    else
                        tma_load_2d_mc(sB + st * kHBBytes + rank * kBPart, &A.tmB, kb * kHK, tn * kHN + rank * (kHN / CL),
                                       &s_full[st], kMask);
                    mbar_arrive(&s_full[st]);
                    if (++st == kHStages) st = 0;
                }
            }
            // every issued load lands before the CTA may leave (the last one of each stage)
            const int lo = it > kHStages ? it - kHStages : 0;
            for (int n = lo; n < it; ++n)
                if (!mbar_wait_bounded(&s_full[n % kHStages], (n / kHStages) & 1)) raise_status(P.status, SPECNG_DEV_TIMEOUT);
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(kHM, kHN);
            int st = 0, it = 0, lt = 0;
            for (int pr = cid; pr < npairs && !*abort_flag; pr += ncl, ++lt) {
                const int b = lt & 1;
                if (lt >= 2 && !mbar_wait_bounded(&s_acce[b], ((lt >> 1) + 1) & 1)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t dt = tmem + b * kHN;
                bool ok = true;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    if (!mbar_wait_bounded(&s_full[st], (it / kHStages) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + st * kHABytes), b0 = smem_u32(sB + st * kHBBytes);
#pragma unroll
                    for (int kk = 0; kk < kHK / 16; ++kk)
                        tc_mma(dt, sdesc_k128(a0 + kk * 32), sdesc_k128(b0 + kk * 32), idesc, (kb | kk) != 0 ? 1u : 0u);
                    // every CTA of the cluster learns when these MMAs have read the stage
                    if constexpr (CL == 1)
                        tc_commit(&s_empty[st]);
                    else
                        tc_commit_mc(&s_empty[st], kMask);
                    if (++st == kHStages) st = 0;
                }
                if (!ok) {
                    give_up();
                    break;
                }
                tc_commit(&s_accf[b]);  // the accumulator is complete
            }
            // every MMA issued has completed before the tensor memory is released
            tc_commit(&s_done);
            if (!mbar_wait_bounded(&s_done, 0)) raise_status(P.status, SPECNG_DEV_TIMEOUT);
        }
        __syncwarp();
    } else {
        // ================= epilogue =================
        const int q = warp & 3;  // the tensor-memory lanes this warp may read: 32 q .. 32 q + 31
        const int V = P.V;
        int last_buf = -1;  // lane 0: staging buffer of the latest committed store (boxes past the data are skipped)
        int lt = 0;
        for (int pr = cid; pr < npairs; pr += ncl, ++lt) {
            const int b = lt & 1;
            if (!mbar_wait_bounded(&s_accf[b], (lt >> 1) & 1)) {
                if (lane == 0) give_up();
                break;
            }
            if (*abort_flag) break;
            tc_fence_after();
            const int tm = CL * (pr % npm) + rank, tn = pr / npm;
            const int row = tm * kHM + 32 * q + lane;
            const bool live = row < A.rows;
            const int v0 = tn * kHN;
            const uint32_t tb = tmem + (static_cast<uint32_t>(32 * q) << 16) + b * kHN;
            const int row0 = tm * kHM + 32 * q;  // the warp's first row
            // one pass: round, store, maxima, and (T > 0) the sum of exponentials against
            // the largest transformed value so far, rescaled when a chunk raises it
            float xmax = -INFINITY, zmax = -INFINITY, s = 0.0f, msc = 0.0f;
            bool bad = false;
#pragma unroll 1
            for (int c0 = 0; c0 < kHN; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tb + c0, r);
                uint32_t w[16];
                float cz = -INFINITY;  // the chunk's largest transformed value
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const float f0 = __uint_as_float(r[i]), f1 = __uint_as_float(r[i + 1]);
                    bad |= !(fabsf(f0) < INFINITY) || !(fabsf(f1) < INFINITY);
                    const uint32_t h0 = bf16_bits(f0), h1 = bf16_bits(f1);
                    w[i >> 1] = h0 | (h1 << 16);
                    const float x0 = __uint_as_float(h0 << 16), x1 = __uint_as_float(h1 << 16);
                    if (v0 + c0 + i < V) {
                        xmax = fmaxf(xmax, x0);
                        if (!GREEDY) cz = fmaxf(cz, transform_f32<SOFTCAP, false>(x0, false, P));
                    }
                    if (v0 + c0 + i + 1 < V) {
                        xmax = fmaxf(xmax, x1);
                        if (!GREEDY) cz = fmaxf(cz, transform_f32<SOFTCAP, false>(x1, false, P));
                    }
                }
                if (c0 + 32 == kHN) {
                    // the last read of this accumulator: it may be overwritten once all four warps are here
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s_acce[b]);
                }
                if (!GREEDY) {
                    if (cz > zmax) {
                        if (zmax > -INFINITY) s *= ex2_approx((zmax - cz) * P.sc);
                        zmax = cz;
                        msc = zmax * P.sc;
                    }
                    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float x = (i & 1) ? __uint_as_float(w[i >> 1] & 0xFFFF0000u) : __uint_as_float(w[i >> 1] << 16);
                        if (v0 + c0 + i < V) acc[i & 3] += ex2_approx(fmaf(sum_transform<SOFTCAP>(x, P), P.sc, -msc));
                    }
                    s += (acc[0] + acc[1]) + (acc[2] + acc[3]);
                }
                // the 32 x 32 box goes out through shared memory with one TMA store
                // (rows past the batch and ids past V are clipped by the store)
                const int bb = (c0 >> 5) & 1;
                uint4* box = s_ep[q][bb];
                // this buffer's previous store has read it: all but the latest committed store
                // are, and the latest too when it used this buffer
                if (lane == 0) {
                    if (last_buf == bb)
                        tma_store_wait_read<0>();
                    else
                        tma_store_wait_read<1>();
                }
                __syncwarp();
#pragma unroll
                for (int u = 0; u < 4; ++u) box[lane * 4 + u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                fence_proxy_async_smem();  // the writes are visible to the TMA unit
                __syncwarp();
                if (lane == 0 && row0 < A.rows && v0 + c0 < V) {
                    tma_store_2d(&A.tmC, v0 + c0, row0, box);
                    last_buf = bb;
                }
            }
            if (__any_sync(0xffffffffu, bad && live) && lane == 0) raise_status(P.status, SPECNG_DEV_NONFINITE);
            if (live) {
                const size_t rec = static_cast<size_t>(row) * P.nblk + tn;
                P.bmax[rec] = xmax;
                if (!GREEDY) P.part[rec] = SegSum{zmax, s};
            }
        }
    }
    if (warp >= 2 && lane == 0) tma_store_wait_all();  // the staged logits are written out
    tc_fence_before();
    __syncthreads();
    // neither CTA leaves while the other may still multicast into it or arrive on its barriers
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kHTmemCols);
    }
}

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once (a thread-safe static).
EncodeTiledFn encode_fn() {
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        return nullptr;
    }();
    return fn;
}

// A [rows, d] bf16 row-major matrix as 64 x box_rows tiles with the 128-byte swizzle.
// The logits [rows, V] bf16 as 32 x 32 boxes, no swizzle (rows of 64 bytes in shared memory).
bool encode_store(CUtensorMap* tm, void* base, int rows, int V) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(V), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(V) * 2};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t es[2] = {1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_k128(CUtensorMap* tm, const void* base, int rows, int d, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kHK), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t es[2] = {1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int CL, bool G, bool C>
cudaError_t launch_lmhead_gc(const LmHeadArgs& A, int ngroups, cudaStream_t s) {
    static bool configured[128] = {};
    static int max_clusters[128] = {};
    bool* done = attr_flag(configured);
    int* mc = max_clusters + (done - configured);
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kHThreads);
    cfg.dynamicSmemBytes = kHSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CL;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    if (!*done) {
        cudaError_t e = cudaFuncSetAttribute(lmhead_verify_kernel<CL, G, C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kHSmem));
        if (e != cudaSuccess) return e;
        int n = sm_count_cached();  // one CTA per SM
        if (CL > 1) {
            // clusters that fit on the device at once (a GPC with an odd number of free SMs
            // leaves one idle): the persistent grid is that many, so there is one wave
            cfg.gridDim = dim3(static_cast<unsigned>(CL * (sm_count_cached() / CL)));
            cfg.attrs = attr + 1;
            cfg.numAttrs = 1;
            e = cudaOccupancyMaxActiveClusters(&n, lmhead_verify_kernel<CL, G, C>, &cfg);
            if (e != cudaSuccess) return e;
            cfg.attrs = attr;
        }
        *mc = n > 0 ? n : 1;
        *done = true;
    }
    cfg.gridDim = dim3(static_cast<unsigned>(CL * std::min(ngroups, *mc)));
    cfg.numAttrs = CL > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, lmhead_verify_kernel<CL, G, C>, A);
}

template <int CL>
cudaError_t launch_lmhead_cl(const LmHeadArgs& A, int ngroups, bool greedy, bool softcap, cudaStream_t s) {
    if (greedy) return softcap ? launch_lmhead_gc<CL, true, true>(A, ngroups, s) : launch_lmhead_gc<CL, true, false>(A, ngroups, s);
    return softcap ? launch_lmhead_gc<CL, false, true>(A, ngroups, s) : launch_lmhead_gc<CL, false, false>(A, ngroups, s);
}

}  // namespace

// Encodes the tensor maps and launches the fused kernel, then the decision
// kernel (and, for dense q at T > 0, the residual pass) on its records.
// Returns cudaErrorInvalidValue when the tensor maps cannot be encoded.
cudaError_t launch_lmhead_verify(const void* hidden, const void* weight, int d, void* logits, VerifyDev P, bool greedy,
                                 bool softcap, bool dense, cudaStream_t s) {
    LmHeadArgs A{};
    const int rows = P.B * (P.K + 1);
    A.rows = rows;
    A.d = d;
    A.ntm = (rows + kHM - 1) / kHM;
    A.ntn = (P.V + kHN - 1) / kHN;
    const int cl = A.ntm % 2 == 0 ? 2 : 1;  // pairs of row tiles when they pair up
    if (!encode_k128(&A.tmA, hidden, rows, d, kHM) || !encode_k128(&A.tmB, weight, P.V, d, kHN / cl) ||
        !encode_store(&A.tmC, logits, rows, P.V))
        return cudaErrorInvalidValue;
    A.logits = static_cast<__nv_bfloat16*>(logits);
    P.logits = logits;
    P.nchunk = P.nblk;  // one record per row and noise block
    A.P = P;
    const int ngroups = A.ntm / cl * A.ntn;
    cudaError_t e = cl == 2 ? launch_lmhead_cl<2>(A, ngroups, greedy, softcap, s)
                            : launch_lmhead_cl<1>(A, ngroups, greedy, softcap, s);
    if (e != cudaSuccess) return e;
    P.records_given = 1;
    return launch_verify_dtype<true>(P, greedy, softcap, false, dense, s);
}

}  // namespace specng
