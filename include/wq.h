/*
 * wq.h -- C ABI of the GB300 W4A16 dequantise-GEMM library (libwq.so).
 *
 * The library computes  C = A . deq(B)^T  on one NVIDIA GB300 (sm_103a):
 *
 *   A        (M, K)   bf16 activations, row-major.
 *   packed   (N, K/2) uint8, a pair of 4-bit codes in each byte; byte j of row n holds
 *            element k = 2j in its LOW nibble and k = 2j+1 in its HIGH
 *            nibble (KBench megakernel_int4_weight_decode.py spec, "The
 *            weight format"; TileLang example_dequant_gemm_bf16_fp4_hopper.py,
 *            simple_dequant_bf16_fp4 indexing).
 *   scales   (N, K/group), one per group of `group` consecutive k of a row:
 *              WQ_NVFP4  float8_e4m3fn bytes, group 16; weight = e2m1(code) *
 *                        |e4m3(scale)| (Matmul2dFp4 Mojo API docs, run /
 *                        run_smem_decode: scales (N, K/16) float8_e4m3fn,
 *                        decode_e2m1 * |scale|);
 *              WQ_MXFP4  e8m0 bytes (2^(E-127), 0xFF = NaN), group 32;
 *                        weight = e2m1(code) * 2^(E-127) (OCP MX; the
 *                        TileLang example applies the same power-of-two
 *                        scale as an exponent offset, _tir_u8_to_f4_to_bf16);
 *              WQ_INT4   bf16 values, any group that is a multiple of 32
 *                        (128 in the KBench spec); weight = (code - zero) *
 *                        scale, the zero point subtracted before the multiply
 *                        (KBench spec, "The weight format" and Precision).
 *            e2m1 codes: 1 sign, 2 exponent (bias 1), 1 mantissa, exponent 0
 *            subnormal: +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}.
 *   zeros    (N, K/group) uint8 zero points for WQ_INT4 (read as full uint8),
 *            NULL for the fp4 formats.
 *   C        (M, N) row-major, bf16 (default) or fp32 (format | WQ_OUT_F32).
 *
 * Accumulation is fp32; bf16 output is rounded to nearest even.
 *
 * Conventions for every entry point:
 *   - All array pointers are DEVICE pointers owned by the caller.  The library
 *     allocates no device memory per call; it keeps only file-scope device
 *     state (a status word) and small per-process host caches.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *     void*, NULL = the legacy default stream); the call returns once it is
 *     enqueued.  Launch failures return WQ_ERR_CUDA; faults during execution
 *     surface at the caller's next synchronisation; a bounded device-side
 *     wait that ran out is reported by wq_get_device_error().
 *   - Shapes: M, N >= 0 (M == 0 or N == 0 is a no-op returning WQ_OK);
 *     K >= 0, a multiple of 32 and of `group`; group as listed above.
 *     Otherwise WQ_ERR_UNSUPPORTED (shape) or WQ_ERR_INVALID_ARG.
 *   - A, packed and C must be 16-byte aligned (WQ_ERR_ALIGN otherwise);
 *     scales 2-byte aligned for WQ_INT4.
 *   - Arguments are validated before anything is launched; no C++ exception
 *     crosses this boundary, and there is no CPU path.
 *   - Calls are thread-safe for distinct streams; calls on one stream run in
 *     order.
 */
#ifndef WQ_H
#define WQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* weight formats: the low byte of `format` */
#define WQ_NVFP4 0
#define WQ_MXFP4 1
#define WQ_INT4 2
/* OR into `format`: write C as fp32 instead of bf16 */
#define WQ_OUT_F32 0x100

/* kernel selection for wq_gemm_ex: the low byte of `path` */
#define WQ_PATH_AUTO 0 /* M <= 16: split-K GEMV; larger M: tensor-core path */
#define WQ_PATH_GEMV 1 /* register-decode GEMV kernel, any M (16 rows per pass) */
#define WQ_PATH_TC 2   /* tcgen05 / TMEM tensor-core kernel */
/* OR into `path`: launch with programmatic dependent launch, so that the
 * GEMV kernel starts streaming its weights while the preceding kernel on the
 * stream is still running (A is read and C written only after that kernel
 * has completed).  The tensor-core kernel takes it for launches of up to two
 * waves of tiles and for split tiles: it sets up (tensor memory, barriers)
 * while its predecessor finishes, and reads A and writes C, partial sums and
 * flags only after that predecessor has completed.  The caller guarantees that the preceding kernel does not
 * write packed, scales, zeros or the prepacked buffer -- true whenever they
 * are model weights, and false right after the wq_prepack that writes them
 * (synchronise first). */
#define WQ_LAUNCH_OVERLAP 0x100
/* OR into `path` (small-M kernels; implies WQ_LAUNCH_OVERLAP): the caller
 * declares that A, like the weights, is written by no kernel that can still
 * be running -- i.e. it was complete before the most recent operation on the
 * stream launched WITHOUT WQ_LAUNCH_OVERLAP / WQ_LAUNCH_INPUTS_READY began.
 * The kernel then reads A and runs its whole product at once, and waits for
 * the preceding kernel only before it stores C, so a chain of such calls
 * (projections that share one input, independent weights of one step)
 * overlaps end to end while still completing in stream order: a later
 * operation on the stream sees the results of every earlier call.  The
 * tensor-core path treats the bit as WQ_LAUNCH_OVERLAP. */
#define WQ_LAUNCH_INPUTS_READY 0x200

/* status codes */
#define WQ_OK 0
#define WQ_ERR_INVALID_ARG (-1)  /* NULL pointer, negative size, bad format/path */
#define WQ_ERR_UNSUPPORTED (-2)  /* shape / group the kernels do not handle */
#define WQ_ERR_ALIGN (-3)        /* pointer alignment */
#define WQ_ERR_CUDA (-4)         /* a CUDA runtime call or launch failed */
#define WQ_ERR_DEVICE_TIMEOUT (-5) /* a bounded device-side wait ran out */

/*
 * wq_gemm -- C = A . deq(packed, scales, zeros)^T on the legacy default
 * stream with automatic kernel selection.  Arguments as in the header
 * comment.  Returns a status code.
 */
int wq_gemm(const void* A, const uint8_t* packed, const void* scales, const uint8_t* zeros,
            void* C, int M, int N, int K, int format, int group);

/*
 * wq_gemm_ex -- wq_gemm on an explicit stream (cudaStream_t as void*) with
 * an explicit kernel choice (WQ_PATH_*, optionally | WQ_LAUNCH_OVERLAP).
 * WQ_PATH_TC returns WQ_ERR_UNSUPPORTED for shapes that kernel does not take
 * (K not a multiple of 64, or row strides not 16-byte aligned for TMA).
 * Where the tensor-core path has so few tiles (128 weight rows x up to 256
 * activation rows) that each can take two or more SMs, it runs each tile on
 * one thread-block cluster of up to 8 CTAs that split the tile's k-steps
 * evenly and add their fp32 partial sums through distributed shared memory,
 * in cluster-rank order (deterministic; no workspace; the method itself has
 * no such step -- it computes the same sum of products).  WQ_TC_CSK in the
 * environment: 0 turns this off, S >= 2 asks for S CTAs per tile (tests).
 */
int wq_gemm_ex(const void* A, const uint8_t* packed, const void* scales, const uint8_t* zeros,
               void* C, int M, int N, int K, int format, int group, void* stream, int path);

/*
 * wq_gemm_ws -- wq_gemm_ex with a caller-owned device workspace that the
 * tensor-core path may use to balance its tiles over the SMs ("stream-K": a
 * tile whose k-steps are shared by two or more CTAs is finished by the CTA
 * holding its last k-step, which adds the fp32 partial sums the others left
 * in the workspace, in a fixed CTA order -- deterministic, no atomics on C).
 * The method itself has no such step: it is a load-balancing device of this
 * library and computes the same sum of products as wq_gemm_ex.
 *   workspace        256-byte aligned device memory (NULL with 0 bytes: the
 *                    call behaves as wq_gemm_ex).  It must hold zeros before
 *                    its first use (cudaMemset).  It starts with one flag
 *                    word per SM, which every completed call leaves zero
 *                    again; the rest holds partial sums that a call always
 *                    writes before it reads them.  So one workspace serves
 *                    any number of calls that are ordered on the device (one
 *                    stream).  After a call that reported
 *                    WQ_ERR_DEVICE_TIMEOUT it must be zeroed again.
 *   workspace_bytes  its size; below wq_gemm_workspace_size() for this shape
 *                    the tiles run whole, as in wq_gemm_ex.
 * Returns WQ_ERR_ALIGN for a misaligned workspace, WQ_ERR_INVALID_ARG for a
 * NULL workspace with a non-zero size.
 */
int wq_gemm_ws(const void* A, const uint8_t* packed, const void* scales, const uint8_t* zeros,
               void* C, int M, int N, int K, int format, int group, void* workspace,
               size_t workspace_bytes, void* stream, int path);

/*
 * wq_gemm_static -- wq_gemm_ws with the library's own scratch instead of a
 * caller-owned workspace: a fixed device array inside the library (room for
 * the split tiles of up to 160 SMs), found once per device, so the call
 * allocates nothing.  The method itself has no such step; it exists so that
 * a caller without a memory allocator still gets the balanced tensor-core
 * path.  Limits: one scratch per device, so calls through this entry point
 * must be ordered on the device (one stream at a time), and a tensor-core
 * call whose split would need more scratch than the array holds returns
 * WQ_ERR_UNSUPPORTED without launching (WQ_STATIC_WS_CAP in the environment
 * lowers the usable size, for tests); calls that run on the small-M kernel
 * use no scratch.  Recovery: a call whose bounded wait ran out leaves flag
 * words set in the scratch; once wq_get_device_error() has returned that
 * WQ_ERR_DEVICE_TIMEOUT, the next wq_gemm_static call on the device first
 * zeroes them with a memset on its stream (nothing is allocated).
 * Otherwise as wq_gemm_ex.
 */
int wq_gemm_static(const void* A, const uint8_t* packed, const void* scales, const uint8_t* zeros,
                   void* C, int M, int N, int K, int format, int group, void* stream, int path);

/*
 * Fused epilogue (the KBench spec's decoder MLP is
 * down(silu(gate(x)) * up(x))).  Every step is optional and runs on the
 * fp32 accumulator of each output element before the cast to C:
 *   y = acc + bias[n]          bias: bf16, one per weight row (N values)
 *   gated: the SiLU-gated product of a gate/up projection pair stored as one
 *          weight of N rows, interleaved in groups of 8: weight rows
 *          16b .. 16b+7 are the gate rows of outputs 8b .. 8b+7 and rows
 *          16b+8 .. 16b+15 their up rows.  Output o = silu(y_gate) * y_up,
 *          silu(x) = x / (1 + e^-x); C then has N / 2 columns (N % 16 == 0,
 *          else WQ_ERR_UNSUPPORTED).
 *   y += residual[m, o]        residual: bf16, row-major, shaped like C
 * bias and residual are device pointers, 2-byte aligned, or NULL.
 */
typedef struct wq_epilogue {
    const void* bias;
    const void* residual;
    int gated; /* 0 or 1 */
} wq_epilogue;

/*
 * wq_gemm_fused -- wq_gemm_ws with a fused epilogue (NULL: none).  N is the
 * number of weight rows.  C is (M, N) or, gated, (M, N / 2).
 */
int wq_gemm_fused(const void* A, const uint8_t* packed, const void* scales, const uint8_t* zeros,
                  void* C, int M, int N, int K, int format, int group, const wq_epilogue* epilogue,
                  void* workspace, size_t workspace_bytes, void* stream, int path);

/* Workspace bytes wq_gemm_ws can use for this shape on the current device
 * (0: the shape needs none -- M <= 16, tiles that fill whole waves, tiles
 * split over thread-block clusters (wq_gemm_ex), or an invalid
 * description). */
size_t wq_gemm_workspace_size(int M, int N, int K, int format, int group);

/* The same size under the name the library's design gives it (an alias of
 * wq_gemm_workspace_size). */
size_t wq_workspace_bytes(int M, int N, int K, int format, int group);

/*
 * Offline repack ("prepack").  The KBench spec's untimed build step may store
 * the weights in whatever layout suits the kernel (nibble order, fragment
 * order, scales apart from the codes) as long as what is streamed per call
 * is still the 4-bit codes.  wq_prepack writes such a
 * layout once; wq_gemm_prepacked then computes the same C as wq_gemm_fused
 * on the original arrays, reading only the prepacked buffer.
 *
 * Formats: WQ_NVFP4 (group 16), WQ_MXFP4 (group 32), WQ_INT4 with group 128.
 * Other int4 groups return WQ_ERR_UNSUPPORTED.
 *
 * Layout (all offsets in bytes from the buffer start; Nb = ceil(N / 16) row
 * blocks, I = ceil(K / 128) k-blocks):
 *   codes    Nb * I blocks of 1024 bytes; block (b, i) at (b * I + i) * 1024
 *            holds rows 16b .. 16b+15 and k = 128i .. 128i+127 as two halves
 *            of 512 bytes, half h (k = 128i + 64h ..) at + 512h.  In a half,
 *            row r (= weight row 16b + r) takes 32 bytes at 32r: eight 4-byte
 *            words w0..w7, w_u holding the 8 codes k0 = 128i + 64h + 8u ..
 *            k0 + 7, stored in the order w0 w4 w1 w5 | w2 w6 w3 w7 and with
 *            the two 16-byte halves of the row exchanged when bit 2 of r is
 *            set.  Inside a word: fp4 keeps the input's byte order (byte j =
 *            k0 + 2j low nibble, k0 + 2j + 1 high nibble); int4 puts k0 + 2s
 *            in nibble s and k0 + 2s + 1 in nibble s + 4 (s = 0..3), so one
 *            mask of the word gives a bf16 pair of consecutive k.  Rows past
 *            N and k past K hold code 0.
 *   records  from Nb * I * 1024, one record block per code block, in the
 *            same order:
 *              WQ_INT4   48 bytes.  Bytes 0..31: row r's bf16 scale at
 *                        4 * (r & 7) + 2 * (r >> 3); bytes 32..47: row r's
 *                        uint8 zero point at 32 + 2 * (r & 7) + (r >> 3)
 *                        (so rows r and r + 8 share one 4-byte and one
 *                        2-byte load).  Rows past N: scale 0, zero 0.
 *              WQ_NVFP4  128 bytes; row r's 8 scale bytes (groups 8i ..
 *                        8i + 7) at 8r.  Groups past K and rows past N: 0.
 *              WQ_MXFP4  64 bytes; row r's 4 scale bytes (groups 4i ..
 *                        4i + 3) at 4r.  Groups past K and rows past N: 0.
 *   flags    WQ_INT4 only: 16 bytes after the last record block; byte 0 is 1
 *            when some zero point exceeds 128 (the kernels then subtract it
 *            in two exact steps, 128 + min(z, 128) and z - min(z, 128)),
 *            else 0; bytes 1..15 are 0.
 */

/* Size in bytes of the prepacked buffer for this weight, 0 for a
 * description wq_prepack does not take (bad or unsupported format or group,
 * K not a multiple of the group, N or K not positive). */
size_t wq_prepack_bytes(int N, int K, int format, int group);

/*
 * wq_prepack -- write the prepacked layout of (packed, scales, zeros) into
 * `prepacked` (device memory, 16-byte aligned, at least wq_prepack_bytes()
 * bytes; every byte of that size is written).  Inputs as for wq_gemm.
 * Asynchronous on `stream`.  Returns WQ_ERR_UNSUPPORTED for descriptions
 * wq_prepack_bytes() gives 0 for, WQ_ERR_INVALID_ARG for a buffer smaller
 * than that size, WQ_ERR_ALIGN for a misaligned buffer or input.
 */
int wq_prepack(const uint8_t* packed, const void* scales, const uint8_t* zeros, void* prepacked,
               size_t prepacked_bytes, int N, int K, int format, int group, void* stream);

/*
 * wq_gemm_prepacked -- C = A . deq(B)^T for a weight B given by its
 * prepacked buffer (N, K, format and group as passed to wq_prepack; format
 * may carry WQ_OUT_F32).  epilogue as for wq_gemm_fused (NULL: none);
 * workspace as for wq_gemm_ws (NULL with 0 bytes: none).  `path`:
 *   WQ_PATH_AUTO  M <= 16: the small-M kernel; larger M: the tensor-core
 *                 kernel (a half block of 8 row blocks is its 128-row weight
 *                 tile), the small-M kernel where that one does not take the
 *                 shape (K not a multiple of 64);
 *   WQ_PATH_GEMV  the small-M kernel for every M (16 activation rows per
 *                 pass; WQ_ERR_UNSUPPORTED for K > 16384);
 *   WQ_PATH_TC    the tensor-core kernel;
 * optionally | WQ_LAUNCH_OVERLAP (small-M kernel).  A and C as for wq_gemm.
 * The buffer must be 16-byte aligned.
 */
int wq_gemm_prepacked(const void* A, const void* prepacked, void* C, int M, int N, int K, int format,
                      int group, const wq_epilogue* epilogue, void* workspace, size_t workspace_bytes,
                      void* stream, int path);

/*
 * wq_dequant -- W = deq(packed, scales, zeros) as an (N, K) row-major bf16
 * matrix, each weight rounded to nearest even from its exact value (so the
 * result equals the oracle's bf16 image bit for bit; NaN stays NaN, overflow
 * goes to +-inf, the sign of zero follows the IEEE product).  W must be
 * 16-byte aligned.  `format` takes no WQ_OUT_F32 flag.
 */
int wq_dequant(const uint8_t* packed, const void* scales, const uint8_t* zeros, void* W,
               int N, int K, int format, int group, void* stream);

/* Returns the device status word (WQ_OK or WQ_ERR_DEVICE_TIMEOUT) of the
 * current device and clears it.  Synchronises the device.  A timeout it
 * returns also marks the library scratch of wq_gemm_static for clearing.
 * Tests can run the tensor-core kernel's failure path on purpose:
 * WQ_TC_FLAG_WAIT_NS in the environment (read at each launch) bounds a
 * stream-K tile owner's wait for its contributors' partial sums, and 0 makes
 * every such wait give up at once; the kernel then unwinds (its copies and
 * MMAs drain under their own bounds), records the timeout and stores
 * nothing for the tiles whose wait gave up. */
int wq_get_device_error(void);

/* Failure-path self test: enqueues a one-thread kernel whose bounded wait on
 * an mbarrier that nothing completes runs out after ~20 ms; the kernel then
 * records WQ_ERR_DEVICE_TIMEOUT exactly as a GEMM kernel would.  Nothing
 * hangs and the context stays usable; wq_get_device_error() afterwards
 * returns (and clears) WQ_ERR_DEVICE_TIMEOUT.  Returns a launch status. */
int wq_selftest_timeout(void* stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* wq_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int wq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* WQ_H */
