// fa_api.cu -- C-ABI entry points of libfa_gb300.so (declared in
// include/fa_gb300.h): argument validation, TMA tensor maps, kernel choice
// and launch.  No device memory is allocated and nothing is synchronised.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa_fwd_kernel.cuh"
#include "fa_gb300.h"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, resolved through the runtime so that the
// library does not link against libcuda.
EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// [B, S, H, D] 16-bit tensor seen as 4-D (D, H, S, B), innermost first; the
// box is 64 elements of D (128 bytes, the 128-byte swizzle span) x 1 head x
// `rows` positions x 1 batch.  Positions past S read as zero and are not
// written by stores.
bool make_map(CUtensorMap* m, const void* base, bool bf16, int B, int S, int H, int D, int rows) {
    EncodeTiledFn enc = encode_tiled();
    if (enc == nullptr) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(H) * D * 2,
                                   static_cast<cuuint64_t>(S) * H * D * 2};
    const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(rows), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r =
        enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D, bool BF16, int NS>
int launch(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int S,
           int causal, float scale, cudaStream_t stream) {
    auto kern = fa::fa_fwd_kernel<D, BF16, NS>;
    constexpr int kSmem = fa::SmemLayout<D, NS>::kAlloc;
    // The dynamic shared-memory opt-in is per device; remember it per device.
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FA_ERR_CUDA;
    std::call_once(once[dev], [&] {
        attr_err[dev] =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    });
    if (attr_err[dev] != cudaSuccess) return FA_ERR_CUDA;

    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, Q, BF16, B, S, H, D, fa::kBM) || !make_map(&mk, K, BF16, B, S, H, D, fa::kBN) ||
        !make_map(&mv, V, BF16, B, S, H, D, fa::kBN) || !make_map(&mo, O, BF16, B, S, H, D, fa::kBM))
        return FA_ERR_CUDA;

    fa::FwdParams p;
    p.B = B;
    p.H = H;
    p.S = S;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    p.lse = LSE;
    const int rows_per_cta = fa::kQTiles * fa::kBM;
    const dim3 grid(static_cast<unsigned>(B) * static_cast<unsigned>(H),
                    static_cast<unsigned>((S + rows_per_cta - 1) / rows_per_cta));
    kern<<<grid, fa::kThreads, kSmem, stream>>>(mq, mk, mv, mo, p);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int validate(const void* Q, const void* K, const void* V, void* O, const float* LSE, int B, int H,
             int S, int D, float scale, int dtype) {
    if (Q == nullptr || K == nullptr || V == nullptr || O == nullptr) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || S < 1) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
                          reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(O);
    if (mis & 15u) return FA_ERR_UNSUPPORTED;
    if (LSE != nullptr && (reinterpret_cast<uintptr_t>(LSE) & 3u)) return FA_ERR_UNSUPPORTED;
    // grid limits: B*H blocks in x, ceil(S / 256) in y (<= 65535)
    const long long rows_per_cta = static_cast<long long>(fa::kQTiles) * fa::kBM;
    if (static_cast<long long>(B) * H > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    if ((static_cast<long long>(S) + rows_per_cta - 1) / rows_per_cta > 65535) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

}  // namespace

extern "C" {

int fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int S,
           int D, int causal, float scale, int dtype, fa_stream_t stream) {
    const int v = validate(Q, K, V, O, LSE, B, H, S, D, scale, dtype);
    if (v != FA_OK) return v;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == FA_F16) {
        if (D == 64) return launch<64, false, 6>(Q, K, V, O, LSE, B, H, S, causal, scale, st);
        return launch<128, false, 4>(Q, K, V, O, LSE, B, H, S, causal, scale, st);
    }
    if (D == 64) return launch<64, true, 6>(Q, K, V, O, LSE, B, H, S, causal, scale, st);
    return launch<128, true, 4>(Q, K, V, O, LSE, B, H, S, causal, scale, st);
}

int fa_fwd_f16(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
               int S, int D, int causal, float scale, fa_stream_t stream) {
    return fa_fwd(Q, K, V, O, LSE, B, H, S, D, causal, scale, FA_F16, stream);
}

int fa_fwd_bf16(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                int S, int D, int causal, float scale, fa_stream_t stream) {
    return fa_fwd(Q, K, V, O, LSE, B, H, S, D, causal, scale, FA_BF16, stream);
}

const char* fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "ok";
        case FA_ERR_INVALID_ARG: return "invalid argument";
        case FA_ERR_UNSUPPORTED: return "unsupported shape, head dimension or alignment";
        case FA_ERR_CUDA: return "CUDA runtime or driver error";
        case FA_ERR_TIMEOUT: return "a device-side wait timed out";
        default: return "unknown status";
    }
}

int fa_device_status(int clear) {
    if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, fa::g_fa_device_status, sizeof(int)) != cudaSuccess)
        return FA_ERR_CUDA;
    if (clear) {
        const int z = 0;
        if (cudaMemcpyToSymbol(fa::g_fa_device_status, &z, sizeof(int)) != cudaSuccess)
            return FA_ERR_CUDA;
    }
    return v;
}

int fa_kernels_per_call(void) { return 1; }

}  // extern "C"
