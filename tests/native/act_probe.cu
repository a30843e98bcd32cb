// GPU probe of the kernels' fast exponential and sigmoid (exp_neg,
// sigmoid_fast in gsa_kernel.cuh): evaluates them, and the SwiGLU value and
// derivatives, at every BF16 bit pattern and writes the FP32 results to
// stdout as raw little-endian floats, in this order:
//   exp_neg(|x|), sigmoid_fast(x), v, da, db of Act<ACT_SWIGLU>::grad(x, 1),
//   sigmoid_val(x), 65536 values each.  One thread per input; every index is below 65536.
#include <cstdio>
#include <vector>

#include "gsa_kernel.cuh"

__global__ void probe(float *out) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= 65536) return;
    const float x = __uint_as_float(static_cast<uint32_t>(i) << 16);
    const gsa::ActP ap{};
    out[i] = gsa::exp_neg(fabsf(x));
    out[65536 + i] = gsa::sigmoid_fast(x);
    float v, da, db;
    gsa::Act<gsa::ACT_SWIGLU>::grad(x, 1.0f, ap, v, da, db);
    out[2 * 65536 + i] = v;
    out[3 * 65536 + i] = da;
    out[4 * 65536 + i] = db;
    out[5 * 65536 + i] = gsa::sigmoid_val(x);
}

int main() {
    const int n = 6 * 65536;
    float *d = nullptr;
    if (cudaMalloc(&d, n * sizeof(float)) != cudaSuccess) return 1;
    probe<<<256, 256>>>(d);
    std::vector<float> h(n);
    if (cudaMemcpy(h.data(), d, n * sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess) return 2;
    cudaFree(d);
    std::fwrite(h.data(), sizeof(float), n, stdout);
    return 0;
}
