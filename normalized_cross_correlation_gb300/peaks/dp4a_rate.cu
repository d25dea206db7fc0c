// dp4a_rate.cu -- throughput of the integer dot product (__dp4a) and, for
// comparison, IMAD and PRMT+IADD on sm_103a: eight independent dependency
// chains per thread, four CTAs of 256 threads per SM, 4096 iterations.
// Prints operations per SM per clock (from clock64) and per second (CUDA
// events).  The ALU roofline of the single-template correlation kernel is
// the dp4a rate times the SM count times the maximum SM clock.
#include <cstdio>
#include <cuda_runtime.h>

template <int OP>
__global__ void probe(unsigned *out, int iters, long long *cycles) {
    unsigned acc[8];
    const unsigned y = 0x01010101u + blockIdx.x;
    for (int c = 0; c < 8; ++c) acc[c] = threadIdx.x * 7u + c;
    const long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            if (OP == 0) acc[c] = __dp4a(acc[c], y, acc[c]);
            else if (OP == 1) acc[c] = acc[c] * y + acc[c];
            else acc[c] = __byte_perm(acc[c], y, 0x4321) + acc[c];
        }
    }
    const long long t1 = clock64();
    unsigned s = 0;
    for (int c = 0; c < 8; ++c) s += acc[c];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

template <int OP>
void run(const char *name, int sms) {
    const int blocks = sms * 4, threads = 256, iters = 4096;
    unsigned *out;
    long long *cyc;
    cudaMalloc(&out, (size_t)blocks * threads * 4);
    cudaMalloc(&cyc, (size_t)blocks * 8);
    probe<OP><<<blocks, threads>>>(out, iters, cyc);
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    cudaEventRecord(a);
    probe<OP><<<blocks, threads>>>(out, iters, cyc);
    cudaEventRecord(b);
    cudaEventSynchronize(b);
    float ms = 0.f;
    cudaEventElapsedTime(&ms, a, b);
    long long mx = 0;
    long long *h = new long long[blocks];
    cudaMemcpy(h, cyc, (size_t)blocks * 8, cudaMemcpyDeviceToHost);
    for (int i = 0; i < blocks; ++i) mx = h[i] > mx ? h[i] : mx;
    delete[] h;
    const double ops = (double)blocks * threads * iters * 8;
    printf("%-9s %.1f ops/clk/SM (clock64)  %.2f Tops/s (events, %.3f ms)  %s\n", name,
           ops / sms / (double)mx, ops / (ms * 1e-3) / 1e12, ms, cudaGetErrorString(cudaGetLastError()));
    cudaFree(out);
    cudaFree(cyc);
}

int main() {
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    run<0>("dp4a", sms);
    run<1>("imad", sms);
    run<2>("prmt+iadd", sms);
    return 0;
}
