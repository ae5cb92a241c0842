// wq_api.cu -- the C ABI (include/wq.h): argument validation and kernel
// selection.  Nothing here computes; every step of the product runs in the
// kernels of wq_dequant.cu, wq_gemv.cu, wq_gemv_tma.cu, wq_tc.cu,
// wq_prepack.cu and wq_gemv_pre.cu.
#include <cstdint>
#include <cstdlib>

#include "wq_internal.h"

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Shared checks of the weight description.  Returns WQ_OK or an error code.
int check_weights(const uint8_t* packed, const void* scales, const uint8_t* zeros, int N, int K,
                  int fmt, int group) {
    if (N < 0 || K < 0) return WQ_ERR_INVALID_ARG;
    if (fmt != WQ_NVFP4 && fmt != WQ_MXFP4 && fmt != WQ_INT4) return WQ_ERR_INVALID_ARG;
    if (group <= 0) return WQ_ERR_INVALID_ARG;
    if (fmt == WQ_NVFP4 && group != 16) return WQ_ERR_UNSUPPORTED;
    if (fmt == WQ_MXFP4 && group != 32) return WQ_ERR_UNSUPPORTED;
    if (fmt == WQ_INT4 && group % 32 != 0) return WQ_ERR_UNSUPPORTED;
    if (K % 32 != 0 || K % group != 0) return WQ_ERR_UNSUPPORTED;
    if (N > 0 && K > 0) {
        if (!packed || !scales) return WQ_ERR_INVALID_ARG;
        if (fmt == WQ_INT4 && !zeros) return WQ_ERR_INVALID_ARG;
        if (fmt != WQ_INT4 && zeros) return WQ_ERR_INVALID_ARG;
        if (!aligned(packed, 16)) return WQ_ERR_ALIGN;
        if (fmt == WQ_INT4 && !aligned(scales, 2)) return WQ_ERR_ALIGN;
    }
    return WQ_OK;
}

}  // namespace

#define WQ_EXPORT __attribute__((visibility("default")))

namespace {

int gemm_impl(const void* A, const uint8_t* packed, const void* scales, const uint8_t* zeros, void* C, int M,
              int N, int K, int format, int group, void* workspace, size_t workspace_bytes, void* stream,
              int path, const wq_epilogue* epi_in = nullptr) {
    if (format & ~(0xFF | WQ_OUT_F32)) return WQ_ERR_INVALID_ARG;
    const int fmt = format & 0xFF;
    const bool out_f32 = (format & WQ_OUT_F32) != 0;
    if (M < 0) return WQ_ERR_INVALID_ARG;
    if (path & ~(0xFF | WQ_LAUNCH_OVERLAP | WQ_LAUNCH_INPUTS_READY)) return WQ_ERR_INVALID_ARG;
    const bool inputs_ready = (path & WQ_LAUNCH_INPUTS_READY) != 0;
    const bool overlap = (path & WQ_LAUNCH_OVERLAP) != 0 || inputs_ready;
    path &= 0xFF;
    if (path != WQ_PATH_AUTO && path != WQ_PATH_GEMV && path != WQ_PATH_TC) return WQ_ERR_INVALID_ARG;
    if (workspace_bytes > 0 && !workspace) return WQ_ERR_INVALID_ARG;
    if (workspace && !aligned(workspace, 256)) return WQ_ERR_ALIGN;
    int st = check_weights(packed, scales, zeros, N, K, fmt, group);
    if (st != WQ_OK) return st;
    if (M == 0 || N == 0) return WQ_OK;
    if (!C || (K > 0 && !A)) return WQ_ERR_INVALID_ARG;
    if (!aligned(C, 16) || (K > 0 && !aligned(A, 16))) return WQ_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (workspace_bytes == 0) workspace = nullptr;
    wq::Epilogue epi{nullptr, nullptr, 0};
    if (epi_in) {
        if (epi_in->gated != 0 && epi_in->gated != 1) return WQ_ERR_INVALID_ARG;
        if (epi_in->gated && N % 16 != 0) return WQ_ERR_UNSUPPORTED;
        if (!aligned(epi_in->bias, 2) || !aligned(epi_in->residual, 2)) return WQ_ERR_ALIGN;
        epi.bias = static_cast<const uint16_t*>(epi_in->bias);
        epi.residual = static_cast<const uint16_t*>(epi_in->residual);
        epi.gated = epi_in->gated;
    }

    if (path == WQ_PATH_TC)
        return wq::launch_tc(A, packed, scales, zeros, C, M, N, K, fmt, group, out_f32, workspace, workspace_bytes,
                             epi, overlap, s);
    if (path == WQ_PATH_AUTO && M > 16 && K > 0) {
        st = wq::launch_tc(A, packed, scales, zeros, C, M, N, K, fmt, group, out_f32, workspace, workspace_bytes,
                           epi, overlap, s);
        if (st != WQ_ERR_UNSUPPORTED) return st;
        // shapes the tensor-core kernel does not take run on the GEMV kernel
    }
    return wq::launch_gemv(A, packed, scales, zeros, C, M, N, K, fmt, group, out_f32, overlap, inputs_ready, epi, s);
}

}  // namespace

extern "C" {

WQ_EXPORT int wq_gemm_ex(const void* A, const uint8_t* packed, const void* scales, const uint8_t* zeros, void* C,
               int M, int N, int K, int format, int group, void* stream, int path) {
    return gemm_impl(A, packed, scales, zeros, C, M, N, K, format, group, nullptr, 0, stream, path);
}

WQ_EXPORT int wq_gemm_ws(const void* A, const uint8_t* packed, const void* scales, const uint8_t* zeros, void* C,
               int M, int N, int K, int format, int group, void* workspace, size_t workspace_bytes, void* stream,
               int path) {
    return gemm_impl(A, packed, scales, zeros, C, M, N, K, format, group, workspace, workspace_bytes, stream, path);
}

WQ_EXPORT int wq_gemm_static(const void* A, const uint8_t* packed, const void* scales, const uint8_t* zeros,
                             void* C, int M, int N, int K, int format, int group, void* stream, int path) {
    // the description first, as every entry point checks it
    if (format & ~(0xFF | WQ_OUT_F32)) return WQ_ERR_INVALID_ARG;
    if (M < 0) return WQ_ERR_INVALID_ARG;
    if (path & ~(0xFF | WQ_LAUNCH_OVERLAP | WQ_LAUNCH_INPUTS_READY)) return WQ_ERR_INVALID_ARG;
    const int route = path & 0xFF;
    if (route != WQ_PATH_AUTO && route != WQ_PATH_GEMV && route != WQ_PATH_TC) return WQ_ERR_INVALID_ARG;
    int st = check_weights(packed, scales, zeros, N, K, format & 0xFF, group);
    if (st != WQ_OK) return st;
    size_t cap = 0;
    void* ws = wq::static_workspace(&cap, static_cast<cudaStream_t>(stream), &st);
    if (!ws) return st != WQ_OK ? st : WQ_ERR_CUDA;
    if (const char* e = getenv("WQ_STATIC_WS_CAP")) {   // tests: a smaller usable part
        const size_t v = (size_t)strtoull(e, nullptr, 10);
        if (v < cap) cap = v;
    }
    // the scratch matters only where the tensor-core kernel runs
    const bool tc = route == WQ_PATH_TC || (route == WQ_PATH_AUTO && M > 16);
    const size_t need = (tc && N > 0 && K > 0 && K % 64 == 0) ? wq::tc_workspace_bytes(M, N, K, format & 0xFF) : 0;
    if (need > cap) return WQ_ERR_UNSUPPORTED;
    return gemm_impl(A, packed, scales, zeros, C, M, N, K, format, group, ws, cap, stream, path);
}

WQ_EXPORT int wq_gemm_fused(const void* A, const uint8_t* packed, const void* scales, const uint8_t* zeros, void* C,
                            int M, int N, int K, int format, int group, const wq_epilogue* epilogue,
                            void* workspace, size_t workspace_bytes, void* stream, int path) {
    return gemm_impl(A, packed, scales, zeros, C, M, N, K, format, group, workspace, workspace_bytes, stream, path,
                     epilogue);
}

WQ_EXPORT size_t wq_gemm_workspace_size(int M, int N, int K, int format, int group) {
    if (M <= 16 || N <= 0 || K <= 0) return 0;
    if (check_weights(reinterpret_cast<const uint8_t*>(16), reinterpret_cast<const void*>(16),
                      (format & 0xFF) == WQ_INT4 ? reinterpret_cast<const uint8_t*>(16) : nullptr, N, K,
                      format & 0xFF, group) != WQ_OK)
        return 0;
    return wq::tc_workspace_bytes(M, N, K, format & 0xFF);
}

WQ_EXPORT size_t wq_workspace_bytes(int M, int N, int K, int format, int group) {
    return wq_gemm_workspace_size(M, N, K, format, group);
}

WQ_EXPORT int wq_gemm(const void* A, const uint8_t* packed, const void* scales, const uint8_t* zeros, void* C, int M,
            int N, int K, int format, int group) {
    return wq_gemm_ex(A, packed, scales, zeros, C, M, N, K, format, group, nullptr, WQ_PATH_AUTO);
}

// prepack takes int4 g128, NVFP4 g16, MXFP4 g32 and positive N, K (K a
// multiple of 32 and of the group, as everywhere)
static bool prepack_desc_ok(int N, int K, int fmt, int group) {
    if (N <= 0 || K <= 0) return false;
    if (check_weights(reinterpret_cast<const uint8_t*>(16), reinterpret_cast<const void*>(16),
                      fmt == WQ_INT4 ? reinterpret_cast<const uint8_t*>(16) : nullptr, N, K, fmt, group) != WQ_OK)
        return false;
    return fmt != WQ_INT4 || group == 128;
}

WQ_EXPORT size_t wq_prepack_bytes(int N, int K, int format, int group) {
    if (format & ~0xFF) return 0;
    return prepack_desc_ok(N, K, format, group) ? wq::prepack_bytes(N, K, format) : 0;
}

WQ_EXPORT int wq_prepack(const uint8_t* packed, const void* scales, const uint8_t* zeros, void* prepacked,
                         size_t prepacked_bytes, int N, int K, int format, int group, void* stream) {
    if (format & ~0xFF) return WQ_ERR_INVALID_ARG;
    int st = check_weights(packed, scales, zeros, N, K, format, group);
    if (st != WQ_OK) return st;
    if (!prepack_desc_ok(N, K, format, group)) return WQ_ERR_UNSUPPORTED;
    if (!prepacked) return WQ_ERR_INVALID_ARG;
    if (prepacked_bytes < wq::prepack_bytes(N, K, format)) return WQ_ERR_INVALID_ARG;
    if (!aligned(prepacked, 16)) return WQ_ERR_ALIGN;
    return wq::launch_prepack(packed, scales, zeros, prepacked, N, K, format, static_cast<cudaStream_t>(stream));
}

WQ_EXPORT int wq_gemm_prepacked(const void* A, const void* prepacked, void* C, int M, int N, int K, int format,
                                int group, const wq_epilogue* epilogue, void* workspace, size_t workspace_bytes,
                                void* stream, int path) {
    if (format & ~(0xFF | WQ_OUT_F32)) return WQ_ERR_INVALID_ARG;
    const int fmt = format & 0xFF;
    if (M < 0 || N < 0 || K < 0) return WQ_ERR_INVALID_ARG;
    if (path & ~(0xFF | WQ_LAUNCH_OVERLAP | WQ_LAUNCH_INPUTS_READY)) return WQ_ERR_INVALID_ARG;
    const bool inputs_ready = (path & WQ_LAUNCH_INPUTS_READY) != 0;
    const bool overlap = (path & WQ_LAUNCH_OVERLAP) != 0 || inputs_ready;
    const int route = path & 0xFF;
    if (route != WQ_PATH_AUTO && route != WQ_PATH_GEMV && route != WQ_PATH_TC) return WQ_ERR_INVALID_ARG;
    if (workspace_bytes > 0 && !workspace) return WQ_ERR_INVALID_ARG;
    if (workspace && !aligned(workspace, 256)) return WQ_ERR_ALIGN;
    if (workspace_bytes == 0) workspace = nullptr;
    if (fmt != WQ_NVFP4 && fmt != WQ_MXFP4 && fmt != WQ_INT4) return WQ_ERR_INVALID_ARG;
    if (group <= 0) return WQ_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return WQ_OK;
    if (!prepack_desc_ok(N, K, fmt, group)) return WQ_ERR_UNSUPPORTED;
    if (!A || !prepacked || !C) return WQ_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(C, 16) || !aligned(prepacked, 16)) return WQ_ERR_ALIGN;
    wq::Epilogue epi{nullptr, nullptr, 0};
    if (epilogue) {
        if (epilogue->gated != 0 && epilogue->gated != 1) return WQ_ERR_INVALID_ARG;
        if (epilogue->gated && N % 16 != 0) return WQ_ERR_UNSUPPORTED;
        if (!aligned(epilogue->bias, 2) || !aligned(epilogue->residual, 2)) return WQ_ERR_ALIGN;
        epi.bias = static_cast<const uint16_t*>(epilogue->bias);
        epi.residual = static_cast<const uint16_t*>(epilogue->residual);
        epi.gated = epilogue->gated;
    }
    const bool out_f32 = (format & WQ_OUT_F32) != 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (route == WQ_PATH_TC)
        return wq::launch_tc_prepacked(A, prepacked, C, M, N, K, fmt, group, out_f32, workspace, workspace_bytes,
                                       epi, overlap, s);
    if (route == WQ_PATH_AUTO && M > 16) {
        const int st = wq::launch_tc_prepacked(A, prepacked, C, M, N, K, fmt, group, out_f32, workspace,
                                               workspace_bytes, epi, overlap, s);
        if (st != WQ_ERR_UNSUPPORTED) return st;
    }
    return wq::launch_gemv_prepacked(A, prepacked, C, M, N, K, fmt, out_f32, overlap, inputs_ready, epi, s);
}

WQ_EXPORT int wq_dequant(const uint8_t* packed, const void* scales, const uint8_t* zeros, void* W, int N, int K,
               int format, int group, void* stream) {
    if (format & ~0xFF) return WQ_ERR_INVALID_ARG;
    const int st = check_weights(packed, scales, zeros, N, K, format, group);
    if (st != WQ_OK) return st;
    if (N == 0 || K == 0) return WQ_OK;
    if (!W) return WQ_ERR_INVALID_ARG;
    if (!aligned(W, 16)) return WQ_ERR_ALIGN;
    return wq::launch_dequant(packed, scales, zeros, W, N, K, format, group, static_cast<cudaStream_t>(stream));
}

WQ_EXPORT int wq_get_device_error(void) {
    const int a = wq::read_and_clear_device_status();
    const int b = wq::read_and_clear_gemv_status();
    const int c = wq::read_and_clear_pre_status();
    const int d = wq::read_and_clear_staged_status();
    return a != 0 ? a : (b != 0 ? b : (c != 0 ? c : d));
}

WQ_EXPORT int wq_selftest_timeout(void* stream) {
    return wq::launch_timeout_selftest(static_cast<cudaStream_t>(stream));
}

WQ_EXPORT const char* wq_status_string(int status) {
    switch (status) {
        case WQ_OK: return "WQ_OK";
        case WQ_ERR_INVALID_ARG: return "WQ_ERR_INVALID_ARG: null pointer, negative size or bad format/path";
        case WQ_ERR_UNSUPPORTED: return "WQ_ERR_UNSUPPORTED: shape or group not handled by the kernels";
        case WQ_ERR_ALIGN: return "WQ_ERR_ALIGN: pointer not aligned as required";
        case WQ_ERR_CUDA: return "WQ_ERR_CUDA: a CUDA runtime call or kernel launch failed";
        case WQ_ERR_DEVICE_TIMEOUT: return "WQ_ERR_DEVICE_TIMEOUT: a bounded device-side wait ran out";
        default: return "unknown wq status";
    }
}

WQ_EXPORT int wq_version(void) { return 100; }

}  // extern "C"
