// silu on the device for a list of bf16 inputs, through the library's own two forms:
// silu_f32 (the activation quantizer's) and silu_f32_nobranch (the fused gate/up
// epilogue's).  Test infrastructure: built and loaded by tests/test_gpu_silu.py.
#include <cuda_runtime.h>

#include <cstdint>

#include "silu.cuh"

namespace {

__global__ void silu_list(const uint16_t* g, float* out, float* out_nb, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float x = nvfp4::bf16_to_f32(g[i]);
    out[i] = nvfp4::silu_f32(x);
    out_nb[i] = nvfp4::silu_f32_nobranch(x);
}

}  // namespace

// host arrays in and out; returns a cudaError_t
extern "C" int device_silu(const uint16_t* g, float* out, float* out_nb, int n) {
    uint16_t* dg = nullptr;
    float* d_out = nullptr;
    cudaError_t e = cudaMalloc(&dg, (size_t)n * 2);
    if (e == cudaSuccess) e = cudaMalloc(&d_out, (size_t)n * 8);
    if (e == cudaSuccess) e = cudaMemcpy(dg, g, (size_t)n * 2, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) {
        silu_list<<<(n + 255) / 256, 256>>>(dg, d_out, d_out + n, n);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaMemcpy(out, d_out, (size_t)n * 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(out_nb, d_out + n, (size_t)n * 4, cudaMemcpyDeviceToHost);
    cudaFree(dg);
    cudaFree(d_out);
    return (int)e;
}
