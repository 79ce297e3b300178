// gdn_conv.cu -- depthwise causal conv1d + SiLU with a K-sample carry state
// (torch-to-nnef page "custom_extractors/gdn", CausalConvUpdateReified: the
// drop-in core of the short convolution in front of the gated delta rule).
//
// Per (b, c), the K carried samples and the S new ones form one sequence x;
//   out_t = SiLU(sum_{i<K} w_i x_{t+1+i})     (the K taps against the window
//                                              that ends at new sample t)
//   final_state = the last K samples of x.
// One thread per (b, c) keeps the window in registers (the kernel length is
// a template parameter, 1 .. 16) and shifts each new sample in; all
// arithmetic is fp32.  The op moves (2K + 2S) elements per
// channel and is bound by memory (decode: S = 1).
#include "gdn_internal.cuh"

namespace gdn {

namespace {

template <typename TI, int K>
__global__ void __launch_bounds__(256)
    causal_conv1d_update_kernel(int64_t BC, int64_t C, int64_t S, const TI* __restrict__ hidden,
                                const TI* conv_state, const TI* __restrict__ weight,
                                TI* __restrict__ out, TI* final_state) {
    const int64_t bc = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (bc >= BC) return;
    const int64_t c = bc % C;
    float w[K], win[K];
#pragma unroll
    for (int i = 0; i < K; ++i) {
        w[i] = ldf(weight + c * K + i);
        win[i] = ldf(conv_state + bc * K + i);
    }
    for (int64_t t = 0; t < S; ++t) {
#pragma unroll
        for (int i = 0; i < K - 1; ++i) win[i] = win[i + 1];
        win[K - 1] = ldf(hidden + bc * S + t);
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < K; ++i) acc = fmaf(w[i], win[i], acc);
        stf(out + bc * S + t, acc / (1.f + expf(-acc)));
    }
    // every read of this channel's carried state happened above, so the new
    // state may overwrite it in place
#pragma unroll
    for (int i = 0; i < K; ++i) stf(final_state + bc * K + i, win[i]);
}

template <typename TI, int K>
void launch_k(int64_t BC, int64_t C, int64_t S, const void* hidden, const void* conv_state,
              const void* weight, void* out, void* final_state, cudaStream_t s) {
    causal_conv1d_update_kernel<TI, K><<<(unsigned)((BC + 255) / 256), 256, 0, s>>>(
        BC, C, S, (const TI*)hidden, (const TI*)conv_state, (const TI*)weight, (TI*)out,
        (TI*)final_state);
}

template <typename TI, int K = 1>
void launch_dispatch(int k, int64_t BC, int64_t C, int64_t S, const void* hidden,
                     const void* conv_state, const void* weight, void* out, void* final_state,
                     cudaStream_t s) {
    if constexpr (K <= kConvMaxK) {
        if (k == K)
            launch_k<TI, K>(BC, C, S, hidden, conv_state, weight, out, final_state, s);
        else
            launch_dispatch<TI, K + 1>(k, BC, C, S, hidden, conv_state, weight, out, final_state, s);
    }
}

}  // namespace

cudaError_t launch_causal_conv1d_update(int64_t B, int64_t C, int64_t S, int K, int dtype,
                                        const void* hidden, const void* conv_state,
                                        const void* weight, void* out, void* final_state,
                                        cudaStream_t s) {
    if (dtype == 1)
        launch_dispatch<__nv_bfloat16>(K, B * C, C, S, hidden, conv_state, weight, out, final_state, s);
    else
        launch_dispatch<float>(K, B * C, C, S, hidden, conv_state, weight, out, final_state, s);
    count_launches(1);
    return cudaPeekAtLastError();
}

}  // namespace gdn
