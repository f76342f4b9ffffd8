// Test program (not part of the library): the library's bounded mbarrier wait,
// on a barrier whose transaction bytes never arrive, must give up after about
// its time limit, report that, and leave the CUDA context usable.
#include <cstdio>

#include "zero_device.cuh"

__global__ void wait_for_nothing(int* ok_out, unsigned long long* ns_out) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        zk::mbar_init(&bar, 1);
        zk::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        zk::mbar_arrive_expect_tx(&bar, 16);  // 16 bytes that no copy will deliver
        const uint64_t t0 = zk::globaltimer_ns();
        const bool ok = zk::mbar_wait_bounded(&bar, 0);
        *ns_out = zk::globaltimer_ns() - t0;
        *ok_out = ok ? 1 : 0;
    }
}

__global__ void count(int* x) { atomicAdd(x, 1); }

int main() {
    int* d = nullptr;
    unsigned long long* dn = nullptr;
    if (cudaMalloc(&d, 8) != cudaSuccess || cudaMalloc(&dn, 8) != cudaSuccess) return 2;
    cudaMemset(d, 0xFF, 8);
    wait_for_nothing<<<1, 32>>>(d, dn);
    const cudaError_t e1 = cudaDeviceSynchronize();
    int ok = -1;
    unsigned long long ns = 0;
    cudaMemcpy(&ok, d, 4, cudaMemcpyDeviceToHost);
    cudaMemcpy(&ns, dn, 8, cudaMemcpyDeviceToHost);
    cudaMemset(d, 0, 4);  // the context is still usable
    count<<<1, 64>>>(d);
    const cudaError_t e2 = cudaDeviceSynchronize();
    int n = 0;
    cudaMemcpy(&n, d, 4, cudaMemcpyDeviceToHost);
    printf("wait_ok=%d elapsed_ns=%llu err1=%d err2=%d counted=%d\n", ok, ns, (int)e1, (int)e2, n);
    return (e1 == cudaSuccess && e2 == cudaSuccess && ok == 0 && n == 64) ? 0 : 1;
}
