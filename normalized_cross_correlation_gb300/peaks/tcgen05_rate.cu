// tcgen05_rate.cu -- rates of tcgen05.mma kind::f16 (f16 operands, fp32
// accumulation in tensor memory, M = 128, K = 16) on sm_103a, for the operand
// layouts the correlation kernels use, and the cost of the hand-offs around
// them.  One CTA issues from one thread; operands are small integers.
//   rate N            K-major A and B, N = 64 / 128 / 256
//   bank              A MN-major over eight shifted copies (both core-matrix
//                     strides 128 bytes), B K-major, N = 128; 1 and 2 CTAs/SM
//   toeplitz          A K-major with 16-byte rows (a template row moves the
//                     descriptor by 16 bytes), B a Hankel buffer (both strides
//                     128 bytes), N = 64; 512 MMAs per tile in rows of 8
//       +commit       a commit to one of 16 mbarriers after every row
//       +ring         a producer warp hands the row buffers over a 16-slot
//                     ring (waits for the commit of the row 16 earlier,
//                     arrives); the issuer waits for each row's barrier
//       +wait         the issuer polls, after every row, a barrier whose
//                     phase completed before the first MMA
//       +wait/8       the same poll after every eighth row only
//       2 issuers     warps 0 and 2 issue alternate rows into accumulators of
//                     their own, each polling the completed barrier after
//                     each of its rows
//   each wait in five forms: mbarrier try_wait (acquire), try_wait.relaxed
//   and test_wait (acquire); a shared-memory word polled with ld.volatile and
//   with ld.acquire (the producer publishes it with st.release); for the
//   ring also named barriers (the producer warp bar.arrive, the issuing warp
//   bar.sync; an 8-slot ring on barriers 1..8)
//   wait              SM cycles of one mbarrier.try_wait on a completed phase
// Every wait is bounded; a wait that runs out sets an error flag.
#include <cstdint>
#include <cstdio>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ uint32_t sa(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
           ((uint64_t)(sbo >> 4) << 32) | (1ull << 46);
}

__device__ __forceinline__ uint32_t try_wait(unsigned long long *b, uint32_t par) {
    uint32_t d;
    asm volatile("{ .reg .pred P; mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2; selp.u32 %0, 1, 0, P; }"
                 : "=r"(d) : "r"(sa(b)), "r"(par) : "memory");
    return d;
}

__device__ __forceinline__ uint32_t try_wait_relaxed(unsigned long long *b, uint32_t par) {
    uint32_t d;
    asm volatile("{ .reg .pred P; mbarrier.try_wait.parity.relaxed.cta.shared::cta.b64 P, [%1], %2; selp.u32 %0, 1, 0, P; }"
                 : "=r"(d) : "r"(sa(b)), "r"(par) : "memory");
    return d;
}

__device__ __forceinline__ uint32_t test_wait(unsigned long long *b, uint32_t par) {
    uint32_t d;
    asm volatile("{ .reg .pred P; mbarrier.test_wait.parity.shared::cta.b64 P, [%1], %2; selp.u32 %0, 1, 0, P; }"
                 : "=r"(d) : "r"(sa(b)), "r"(par) : "memory");
    return d;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *f) {
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(sa(f)) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_volatile(const uint32_t *f) {
    uint32_t v;
    asm volatile("ld.volatile.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(sa(f)) : "memory");
    return v;
}

// the flag forms: wait until the word reaches `target`
template <int WAIT>
__device__ __forceinline__ bool flag_bounded(const uint32_t *f, uint32_t target) {
    for (unsigned spin = 0; spin < (1u << 24); ++spin)
        if ((WAIT == 3 ? ld_volatile(f) : ld_acquire(f)) >= target) return true;
    return false;
}

// WAIT: 0 try_wait (acquire), 1 try_wait.relaxed, 2 test_wait (acquire)
template <int WAIT = 0>
__device__ __forceinline__ bool wait_bounded(unsigned long long *b, uint32_t par) {
    for (unsigned spin = 0; spin < (1u << 24); ++spin)
        if (WAIT == 0 ? try_wait(b, par) : WAIT == 1 ? try_wait_relaxed(b, par) : test_wait(b, par)) return true;
    return false;
}

__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
                 ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

__device__ __forceinline__ void commit(unsigned long long *b) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(sa(b)) : "memory");
}

constexpr int kRing = 16;
constexpr int kHRows = 184, kHBytes = kHRows * 16;  // Hankel buffer for K = 128
constexpr int kR = 192;                             // A rows of a Toeplitz tile

// KIND: 0 rate (N), 1 bank, 2 toeplitz, 3 toeplitz+commit, 4 toeplitz+ring,
// 5 toeplitz+wait; WAIT: the form of the issuer's waits (kinds 4 and 5)
template <int KIND, int N, int WAIT = 0>
__global__ void rate_kernel(long long *cyc, int nmma, int *err) {
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ uint32_t taddr_s;
    __shared__ __align__(8) unsigned long long done_bar, ready_bar, full[kRing], empty[kRing];
    __shared__ uint32_t ready_flag, full_flag[kRing];
    const int tid = threadIdx.x, warp = tid >> 5;
    const bool toep = KIND >= 2;
    // operand regions: A first, then B
    const int aBytes = toep ? 16 * kR * 16 : KIND == 1 ? 8 * 2176 : 128 * 32;
    const int bBytes = toep ? kRing * kHBytes : N * 32;
    unsigned char *A = sm, *B = sm + ((aBytes + 1023) / 1024) * 1024;
    for (int i = tid; i < aBytes / 2; i += blockDim.x)
        ((__half *)A)[i] = __float2half((float)((int)((i * 2654435761u) >> 25) - 64));
    for (int i = tid; i < bBytes / 2; i += blockDim.x)
        ((__half *)B)[i] = __float2half((float)((int)((i * 40503u) >> 9 & 127) - 64));
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sa(&done_bar)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sa(&ready_bar)));
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sa(&ready_bar)) : "memory");
        ready_flag = 1;
        for (int i = 0; i < kRing; ++i) full_flag[i] = 0;
        for (int i = 0; i < kRing; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sa(&full[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sa(&empty[i])));
        }
        asm volatile("fence.mbarrier_init.release.cluster;");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    constexpr uint32_t cols = KIND == 6 ? 512 : toep ? 256 : (N < 32 ? 32 : N);
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(sa(&taddr_s)), "r"(cols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    const uint32_t tm = taddr_s;
    constexpr int ring = WAIT == 5 ? 8 : kRing;
    if (KIND == 6 && (warp == 0 || warp == 2) && (tid & 31) == 0) {
        // two issuing threads, alternate rows, separate accumulators
        const int w = warp >> 1;
        const long long t0 = clock64();
        const uint32_t idesc = (1u << 4) | ((uint32_t)(64 >> 3) << 17) | ((128u >> 4) << 24);
        const uint64_t a0 = desc(sa(A), kR * 16, 128), h0 = desc(sa(B), 128, 128);
        for (int q = w; q * 8 < nmma; q += 2) {
            const int j = q & 63, slot = q % kRing;
            const uint32_t d = tm + (uint32_t)w * 256 + (uint32_t)(j >> 4) * 64;
            for (int c = 0; c < 8; ++c)
                mma(d, a0 + (uint64_t)((j * 16 + c * 2 * kR * 16) >> 4),
                    h0 + (uint64_t)((slot * kHBytes + c * 256) >> 4), idesc, ((j & 15) > 1 || c != 0) ? 1u : 0u);
            if (!wait_bounded<WAIT>(&ready_bar, 0)) atomicExch(err, 4);
        }
        unsigned long long *bar = w ? &empty[0] : &done_bar;
        commit(bar);
        if (!wait_bounded(bar, 0)) atomicExch(err, 1);
        if (w == 0) cyc[blockIdx.x] = clock64() - t0;
    } else if (KIND == 6) {
    } else if (KIND == 4 && WAIT == 5 && warp == 0) {
        // the whole issuing warp takes the named barrier; lane 0 issues
        const long long t0 = clock64();
        const uint32_t idesc = (1u << 4) | ((uint32_t)(64 >> 3) << 17) | ((128u >> 4) << 24);
        const uint64_t a0 = desc(sa(A), kR * 16, 128), h0 = desc(sa(B), 128, 128);
        for (int q = 0; q * 8 < nmma; ++q) {
            const int j = q & 63, slot = q % ring;
            asm volatile("bar.sync %0, 64;" ::"r"(1 + slot) : "memory");
            if (tid == 0) {
                const uint32_t d = tm + (uint32_t)(j >> 4) * 64;
                for (int c = 0; c < 8; ++c)
                    mma(d, a0 + (uint64_t)((j * 16 + c * 2 * kR * 16) >> 4),
                        h0 + (uint64_t)((slot * kHBytes + c * 256) >> 4), idesc,
                        ((j & 15) != 0 || c != 0) ? 1u : 0u);
                commit(&empty[slot]);
            }
            __syncwarp();
        }
        if (tid == 0) {
            commit(&done_bar);
            if (!wait_bounded(&done_bar, 0)) atomicExch(err, 1);
            cyc[blockIdx.x] = clock64() - t0;
        }
        __syncwarp();
    } else if (KIND == 4 && WAIT == 5 && warp == 1) {
        // producer warp: slot q's buffer is free once the commit of row q-8
        // landed; a wait that runs out flags the error and still arrives, so
        // the issuing warp's bar.sync always completes
        for (int q = 0; q * 8 < nmma; ++q) {
            const int slot = q % ring;
            if (tid == 32 && q >= ring && !wait_bounded(&empty[slot], ((q / ring) - 1) & 1)) atomicExch(err, 3);
            __syncwarp();
            asm volatile("bar.arrive %0, 64;" ::"r"(1 + slot) : "memory");
        }
    } else if (tid == 0) {
        const long long t0 = clock64();
        if (!toep) {
            // D f32; A MN-major for the bank layout (bit 15); B K-major; N; M = 128
            const uint32_t idesc = (1u << 4) | ((KIND == 1 ? 1u : 0u) << 15) |
                                   ((uint32_t)(N >> 3) << 17) | ((128u >> 4) << 24);
            const uint64_t a0 = KIND == 1 ? desc(sa(A), 128, 128) : desc(sa(A), 2048, 128);
            const uint64_t b0 = desc(sa(B), N * 16, 128);
            uint32_t s = 0;
            for (int i = 0; i < nmma; ++i) {
                mma(tm, a0 + (uint64_t)(KIND == 1 ? s * (2176 >> 4) : 0), b0, idesc, i ? 1u : 0u);
                if (++s == 8) s = 0;
            }
        } else {
            const uint32_t idesc = (1u << 4) | ((uint32_t)(64 >> 3) << 17) | ((128u >> 4) << 24);
            const uint64_t a0 = desc(sa(A), kR * 16, 128), h0 = desc(sa(B), 128, 128);
            for (int q = 0; q * 8 < nmma; ++q) {  // q: template row (8 MMAs)
                const int j = q & 63, slot = q % ring;
                if (KIND == 4 && WAIT < 5 &&
                    !(WAIT < 3 ? wait_bounded<WAIT>(&full[slot], (q / ring) & 1)
                               : flag_bounded<WAIT>(&full_flag[slot], (uint32_t)q + 1)))
                    atomicExch(err, 2);
                const uint32_t d = tm + (uint32_t)(j >> 4) * 64;
                for (int c = 0; c < 8; ++c)
                    mma(d, a0 + (uint64_t)((j * 16 + c * 2 * kR * 16) >> 4),
                        h0 + (uint64_t)((slot * kHBytes + c * 256) >> 4), idesc,
                        ((j & 15) != 0 || c != 0) ? 1u : 0u);
                if (KIND == 3 || KIND == 4) commit(&empty[slot]);
                if ((KIND == 5 || (KIND == 7 && (q & 7) == 7)) && !(WAIT < 3 ? wait_bounded<WAIT>(&ready_bar, 0) : flag_bounded<WAIT>(&ready_flag, 1)))
                    atomicExch(err, 4);
            }
        }
        commit(&done_bar);
        if (!wait_bounded(&done_bar, 0)) atomicExch(err, 1);
        cyc[blockIdx.x] = clock64() - t0;
    } else if (KIND == 4 && tid == 32) {
        // producer: row q's buffer is free once the commit of row q-16 landed
        for (int q = 0; q * 8 < nmma; ++q) {
            const int slot = q % ring;
            if (q >= ring && !wait_bounded(&empty[slot], ((q / ring) - 1) & 1)) {
                atomicExch(err, 3);
                break;
            }
            if (WAIT < 3)
                asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sa(&full[slot])) : "memory");
            else
                asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(sa(&full_flag[slot])), "r"(q + 1)
                             : "memory");
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tm), "r"(cols));
}

// The bank kernel's accumulator pattern on its operand layout (N = 128, A
// MN-major over shifted copies): chains of `chain` MMAs, the first of each
// overwriting its accumulator, accumulators alternating over `stages`
// stages of 128 columns starting at column `dcol` of a 512-column
// allocation (one CTA per SM).
__global__ void bank_pattern(long long *cyc, int nmma, int chain, int stages, int dcol, int *err) {
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ uint32_t taddr_s;
    __shared__ __align__(8) unsigned long long done_bar;
    const int tid = threadIdx.x, warp = tid >> 5;
    unsigned char *A = sm, *B = sm + 18432;
    for (int i = tid; i < 8 * 2176 / 2; i += blockDim.x)
        ((__half *)A)[i] = __float2half((float)((int)((i * 2654435761u) >> 25) - 64));
    for (int i = tid; i < 128 * 32 / 2; i += blockDim.x)
        ((__half *)B)[i] = __float2half((float)((int)((i * 40503u) >> 9 & 127) - 64));
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sa(&done_bar)));
        asm volatile("fence.mbarrier_init.release.cluster;");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(sa(&taddr_s)), "r"(512u));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    const uint32_t tm = taddr_s;
    if (tid == 0) {
        const long long t0 = clock64();
        const uint32_t idesc = (1u << 4) | (1u << 15) | ((uint32_t)(128 >> 3) << 17) | ((128u >> 4) << 24);
        const uint64_t a0 = desc(sa(A), 128, 128), b0 = desc(sa(B), 2048, 128);
        uint32_t s = 0, k = 0, st = 0;
        for (int i = 0; i < nmma; ++i) {
            mma(tm + (uint32_t)dcol + st * 128u, a0 + (uint64_t)(s * (2176 >> 4)), b0, idesc, k ? 1u : 0u);
            if (++s == 8) s = 0;
            if (++k == (uint32_t)chain) {
                k = 0;
                if (++st == (uint32_t)stages) st = 0;
            }
        }
        commit(&done_bar);
        if (!wait_bounded(&done_bar, 0)) atomicExch(err, 1);
        cyc[blockIdx.x] = clock64() - t0;
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tm), "r"(512u));
}

void run_bank_pattern(int sms, int chain, int stages, int dcol) {
    const int nmma = 8192 / chain * chain, smem = 120 * 1024;  // one CTA per SM (512 TMEM columns)
    cudaFuncSetAttribute(bank_pattern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    long long *cyc;
    int *err;
    cudaMalloc(&cyc, (size_t)sms * 8);
    cudaMalloc(&err, 4);
    cudaMemset(err, 0, 4);
    bank_pattern<<<sms, 128, smem>>>(cyc, nmma, chain, stages, dcol, err);
    bank_pattern<<<sms, 128, smem>>>(cyc, nmma, chain, stages, dcol, err);
    long long *h = new long long[sms];
    cudaMemcpy(h, cyc, (size_t)sms * 8, cudaMemcpyDeviceToHost);
    long long mx = 0;
    for (int i = 0; i < sms; ++i) mx = h[i] > mx ? h[i] : mx;
    delete[] h;
    int he = 0;
    cudaMemcpy(&he, err, 4, cudaMemcpyDeviceToHost);
    printf("bank pattern     chain %2d, %d stage(s) from column %3d: %6.1f SM cycles per MMA  err=%d %s\n",
           chain, stages, dcol, (double)mx / nmma, he, cudaGetErrorString(cudaGetLastError()));
    cudaFree(cyc);
    cudaFree(err);
}

// The bank kernel's operand geometry at two CTAs per SM: A over a ring of
// `aslots` slots of 2176 bytes (one per image row, advancing per MMA), B
// (N = 128: two 64-template blocks) with its K halves `blbo` bytes apart and
// its window moving by 1 KB per MMA over 17 positions; chains of 17 MMAs
// alternating over two 128-column accumulators.
__global__ void bank_geometry(long long *cyc, int nmma, int aslots, int blbo, int bmove, int *err) {
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ uint32_t taddr_s;
    __shared__ __align__(8) unsigned long long done_bar;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int bBytes = blbo + 2048 + 17 * 1024;   // the moving window's reach, both K halves
    unsigned char *B = sm, *A = sm + ((bBytes + 1023) / 1024) * 1024;
    for (int i = tid; i < aslots * 2176 / 2; i += blockDim.x)
        ((__half *)A)[i] = __float2half((float)((int)((i * 2654435761u) >> 25) - 64));
    for (int i = tid; i < bBytes / 2; i += blockDim.x)
        ((__half *)B)[i] = __float2half((float)((int)((i * 40503u) >> 9 & 127) - 64));
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sa(&done_bar)));
        asm volatile("fence.mbarrier_init.release.cluster;");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(sa(&taddr_s)), "r"(256u));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    const uint32_t tm = taddr_s;
    if (tid == 0) {
        const long long t0 = clock64();
        const uint32_t idesc = (1u << 4) | (1u << 15) | ((uint32_t)(128 >> 3) << 17) | ((128u >> 4) << 24);
        const uint64_t a0 = desc(sa(A), 128, 128), b0 = desc(sa(B), (uint32_t)blbo, 128);
        uint32_t s = 0, k = 0, st = 0;
        for (int i = 0; i < nmma; ++i) {
            const uint32_t win = bmove ? (16u - k) * (1024u >> 4) : 0u;
            mma(tm + st * 128u, a0 + (uint64_t)(s * (2176 >> 4)), b0 + win, idesc, k ? 1u : 0u);
            if (++s == (uint32_t)aslots) s = 0;
            if (++k == 17u) {
                k = 0;
                st ^= 1u;
            }
        }
        commit(&done_bar);
        if (!wait_bounded(&done_bar, 0)) atomicExch(err, 1);
        cyc[blockIdx.x] = clock64() - t0;
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tm), "r"(256u));
}

void run_bank_geometry(int sms, int ctas, int aslots, int blbo, int bmove) {
    const int blocks = sms * ctas, nmma = 17 * 480, smem = 110 * 1024;  // B reach + 32 A slots = 105 KB
    cudaFuncSetAttribute(bank_geometry, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    long long *cyc;
    int *err;
    cudaMalloc(&cyc, (size_t)blocks * 8);
    cudaMalloc(&err, 4);
    cudaMemset(err, 0, 4);
    bank_geometry<<<blocks, 128, smem>>>(cyc, nmma, aslots, blbo, bmove, err);
    bank_geometry<<<blocks, 128, smem>>>(cyc, nmma, aslots, blbo, bmove, err);
    long long *h = new long long[blocks];
    cudaMemcpy(h, cyc, (size_t)blocks * 8, cudaMemcpyDeviceToHost);
    long long mx = 0;
    for (int i = 0; i < blocks; ++i) mx = h[i] > mx ? h[i] : mx;
    delete[] h;
    int he = 0;
    cudaMemcpy(&he, err, 4, cudaMemcpyDeviceToHost);
    printf("bank geometry    %d CTA(s)/SM, %2d A slots, B K halves %5d B apart%s: %6.1f SM cycles per MMA per CTA  err=%d %s\n",
           ctas, aslots, blbo, bmove ? ", moving window" : "", (double)mx / nmma, he,
           cudaGetErrorString(cudaGetLastError()));
    cudaFree(cyc);
    cudaFree(err);
}

// SM cycles of a try_wait on a phase that completed long before
__global__ void wait_cost(long long *out) {
    __shared__ __align__(8) unsigned long long b;
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sa(&b)));
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sa(&b)) : "memory");
        uint32_t sum = 0;
        const long long t0 = clock64();
        for (int i = 0; i < 64; ++i) sum += try_wait(&b, 0);
        const long long t1 = clock64();
        out[0] = (t1 - t0) / 64;
        out[1] = sum;
    }
}

template <int KIND, int N, int WAIT = 0>
void run(const char *name, int sms, int ctasPerSm) {
    const int blocks = sms * ctasPerSm, nmma = 8192;
    const int smem = 64 * 1024 + (KIND >= 2 ? 64 * 1024 : 0);
    cudaFuncSetAttribute(rate_kernel<KIND, N, WAIT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    long long *cyc;
    int *err;
    cudaMalloc(&cyc, (size_t)blocks * 8);
    cudaMalloc(&err, 4);
    cudaMemset(err, 0, 4);
    rate_kernel<KIND, N, WAIT><<<blocks, 128, smem>>>(cyc, nmma, err);
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    cudaEventRecord(a);
    rate_kernel<KIND, N, WAIT><<<blocks, 128, smem>>>(cyc, nmma, err);
    cudaEventRecord(b);
    cudaEventSynchronize(b);
    float ms = 0.f;
    cudaEventElapsedTime(&ms, a, b);
    long long *h = new long long[blocks];
    cudaMemcpy(h, cyc, (size_t)blocks * 8, cudaMemcpyDeviceToHost);
    long long mx = 0;
    for (int i = 0; i < blocks; ++i) mx = h[i] > mx ? h[i] : mx;
    delete[] h;
    int he = 0;
    cudaMemcpy(&he, err, 4, cudaMemcpyDeviceToHost);
    const int n = KIND >= 2 ? 64 : N;
    const double flops = 2.0 * 128 * n * 16 * (double)nmma * blocks;
    printf("%-16s N=%3d CTAs/SM=%d: %6.1f SM cycles per MMA per CTA  %7.1f TFLOP/s  err=%d %s\n", name, n,
           ctasPerSm, (double)mx / nmma, flops / (ms * 1e-3) / 1e12, he,
           cudaGetErrorString(cudaGetLastError()));
    cudaFree(cyc);
    cudaFree(err);
}

}  // namespace

int main() {
    setvbuf(stdout, NULL, _IONBF, 0);
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    run<0, 64>("rate", sms, 1);
    run<0, 128>("rate", sms, 1);
    run<0, 256>("rate", sms, 1);
    run<1, 128>("bank", sms, 1);
    run<1, 128>("bank", sms, 2);
    run<2, 64>("toeplitz", sms, 1);
    run<3, 64>("toeplitz+commit", sms, 1);
    run<4, 64, 0>("toeplitz+ring", sms, 1);
    run<4, 64, 1>("+ring relaxed", sms, 1);
    run<4, 64, 2>("+ring test_wait", sms, 1);
    run<5, 64, 0>("toeplitz+wait", sms, 1);
    run<5, 64, 1>("+wait relaxed", sms, 1);
    run<5, 64, 2>("+wait test_wait", sms, 1);
    run<4, 64, 3>("+ring ld.volatile", sms, 1);
    run<4, 64, 4>("+ring ld.acquire", sms, 1);
    run<5, 64, 3>("+wait ld.volatile", sms, 1);
    run<5, 64, 4>("+wait ld.acquire", sms, 1);
    run<4, 64, 5>("+ring bar.sync", sms, 1);
    run<7, 64, 0>("+wait/8", sms, 1);
    run<6, 64, 0>("2 issuers+wait", sms, 1);
    run_bank_pattern(sms, 8192, 1, 0);
    run_bank_pattern(sms, 8192, 1, 256);
    run_bank_pattern(sms, 17, 1, 0);
    run_bank_pattern(sms, 17, 2, 0);
    run_bank_pattern(sms, 17, 2, 256);
    run_bank_geometry(sms, 1, 8, 2048, 0);
    run_bank_geometry(sms, 2, 8, 2048, 0);
    run_bank_geometry(sms, 2, 32, 2048, 0);
    run_bank_geometry(sms, 2, 32, 18432, 0);
    run_bank_geometry(sms, 2, 32, 18432, 1);
    run_bank_geometry(sms, 1, 32, 18432, 1);
    long long *w;
    cudaMalloc(&w, 16);
    wait_cost<<<1, 32>>>(w);
    long long hw[2] = {0, 0};
    cudaMemcpy(hw, w, 16, cudaMemcpyDeviceToHost);
    printf("wait             try_wait on a completed phase: %lld SM cycles (%s)\n", hw[0],
           cudaGetErrorString(cudaGetLastError()));
    cudaFree(w);
    return 0;
}
