/*
 * zs.h -- C ABI of libzs: the zonal scatter of the geometric initial
 * embedding (GIE) of an SO(3)-equivariant interatomic potential, lmax = 3,
 * forward and backward, with the stable destination CSR it walks.
 *
 * What the operation is: deepmd-kit pull request "fused Triton zonal scatter
 * for the GIE head (DP_GIE_SCATTER_INFER)", section "What" (forward bullet:
 * a node-parallel walk of the stable destination CSR that accumulates the
 * message without materialising the (E, D-1, C) surface and writes the
 * padded (N, D, C) node layout with a zero scalar row; backward bullet: one
 * edge-parallel pass giving the (E, D-1) coupling and (E, lmax, C) radial
 * gradients; last bullet: the reduction follows the stable-sort CSR order)
 * and section "Boundary and layout contract" (contiguous inputs, the packed
 * lmax = 3 row layout of degree groups 3/5/7).
 *
 * Notation: D = 16 node rows, R = 15 zonal rows, rows 0..2 are degree 1,
 * rows 3..7 degree 2, rows 8..14 degree 3; radial slot s = degree - 1.
 *   coup  (E, 15)     fp32, row-major, contiguous
 *   rad   (E, 3, C)   fp32, row-major, contiguous
 *   out   (N, 16, C)  fp32, row-major, contiguous
 *   g     (N, 16, C)  fp32 cotangent of out (row 0 is never read)
 * Every entry point with an lmax argument also takes the other ladders
 * lmax = 1..5 (an extension of the pages' operator, same definitions):
 * D = (lmax+1)^2, R = D - 1, degree l holding rows [l^2 - 1, (l+1)^2 - 1),
 * coup (E, R), rad (E, lmax, C), out and g (N, D, C).  C = 32 with 16-byte
 * aligned operands takes the vectorised kernels at every lmax (tuned at
 * lmax = 3); every other shape takes per-channel kernels.
 *   forward:  out[n,0,c] = 0,
 *             out[n,1+r,c] = sum over CSR positions j of node n, in order,
 *                            of coup[e,r] * rad[e,s(r),c], e = perm[j]
 *   backward: d_coup[e,r]  = sum_c g[dst[e],1+r,c] * rad[e,s(r),c]
 *             d_rad[e,s,c] = sum over rows r of slot s of g[dst[e],1+r,c] * coup[e,r]
 *
 * Conventions for every entry point:
 *   - All array pointers are DEVICE pointers owned by the caller.  Inputs are
 *     only read.  Outputs are fully overwritten (the caller need not zero
 *     them).  The library never allocates or frees memory; scratch comes from
 *     the caller's workspace, sized by the matching *_workspace_bytes query.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and is asynchronous: no entry point synchronises the
 *     host.  A status other than ZS_OK means nothing was enqueued, except
 *     ZS_ERR_CUDA, which reports a failed launch (see zs_last_error()).
 *   - E = 0 and N = 0 are valid.  Sizes are limited to E < 2^31 (perm and
 *     row_ptr are int32); all address arithmetic inside is 64-bit.
 *   - Results are bitwise deterministic run to run for the same inputs.
 *   - Destinations outside [0, N) belong to no node (reading of the pages,
 *     which leave them undefined): the CSR build counts them and places them
 *     after all valid edges; the backward gives those edges zero gradients.
 *   - Operands are contiguous row-major arrays (the coupling rows may be
 *     strided through the *_ld entry points).  As on the pages, where the
 *     inputs are flattened to contiguous before they enter the operator, a
 *     caller holding a sliced view of the radial operand makes it
 *     contiguous first; the PyTorch operators over this library do that.
 *   - Any C >= 1 is accepted.  C == 32 with 16-byte aligned float4 operands
 *     (rad and out in the forward; g, rad and d_rad in the backward) takes
 *     the vectorised path; every other case takes a per-channel path with
 *     the same results up to fp32 rounding order.
 */
#ifndef ZS_H_
#define ZS_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ZS_API __attribute__((visibility("default")))
#else
#define ZS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, spelled without the CUDA headers. */
typedef struct CUstream_st* zs_stream_t;

typedef enum zs_status {
    ZS_OK = 0,
    ZS_ERR_INVALID_ARG = 1,  /* null pointer with nonzero size, negative size, E >= 2^31, C < 1, workspace too small */
    ZS_ERR_UNSUPPORTED = 2,  /* lmax outside 1..5 */
    ZS_ERR_CUDA = 3,         /* a CUDA call or launch failed; zs_last_error() has the message */
    ZS_ERR_TIMEOUT = 4       /* a bounded device wait ran out (see zs_check_timeouts) */
} zs_status;

/* Static, human-readable name of a status code. */
ZS_API const char* zs_status_string(int status);

/* Message of the last ZS_ERR_* returned on the calling host thread ("" if none). */
ZS_API const char* zs_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
ZS_API int zs_version(void);

/*
 * Bytes of device workspace zs_build_csr needs for E edges and N nodes
 * (0 when E == 0).  The workspace must be 256-byte aligned.
 */
ZS_API size_t zs_build_csr_workspace_bytes(int64_t E, int32_t N);

/*
 * Stable destination CSR ("stable-sort CSR order", pull request "fused
 * Triton zonal scatter for the GIE head", section "What").
 *   dst            (E,)   int32 destination node of each edge
 *   row_ptr        (N+1,) int32 out: node n owns CSR positions [row_ptr[n], row_ptr[n+1])
 *   perm           (E,)   int32 out: edge id at each CSR position; within a node,
 *                         edge ids ascend (stable); edges with dst outside [0, N)
 *                         fill positions [row_ptr[N], E) in ascending edge order
 *   bad_dst_count  (1,)   int32 out, may be NULL: number of edges with dst outside [0, N)
 *   workspace             device scratch of zs_build_csr_workspace_bytes(E, N) bytes
 * The result is bit-identical to a sequential counting sort.
 */
ZS_API zs_status zs_build_csr(const int32_t* dst, int64_t E, int32_t N,
                       int32_t* row_ptr, int32_t* perm, int32_t* bad_dst_count,
                       void* workspace, size_t workspace_bytes, zs_stream_t stream);

/*
 * Bytes of device workspace zs_forward needs at lmax = 3 (partial sums of
 * nodes whose edges are split across work units, and flags that mark them
 * written).  256-byte alignment required; its contents need not start at
 * zero.
 */
ZS_API size_t zs_forward_workspace_bytes(int64_t E, int32_t N, int32_t C);

/*
 * The same for any ladder lmax = 1..5 (0 for an lmax outside that range);
 * equal to zs_forward_workspace_bytes at lmax = 3.
 */
ZS_API size_t zs_forward_workspace_bytes_lmax(int64_t E, int32_t N, int32_t C, int32_t lmax);

/*
 * Forward zonal scatter (pull request "fused Triton zonal scatter for the
 * GIE head", section "What", forward bullet).
 *   coup (E,15), rad (E,3,C)  inputs, indexed by edge id
 *   row_ptr (N+1,), perm (E,) a CSR as produced by zs_build_csr; positions
 *                             row_ptr[N]..E-1 are ignored
 *   E                         length of perm and number of rows of coup/rad
 *   lmax                      1..5 (else ZS_ERR_UNSUPPORTED); the workspace is
 *                             zs_forward_workspace_bytes_lmax(E, N, C, lmax)
 *   out (N,16,C)              output, fully written: row 0 and the rows of
 *                             nodes without edges are exact zeros
 * Each node's sum is formed in fp32 in a fixed order: CSR order within
 * fixed windows of positions, windows combined in ascending order.
 */
ZS_API zs_status zs_forward(const float* coup, const float* rad,
                     const int32_t* row_ptr, const int32_t* perm,
                     int64_t E, int32_t N, int32_t C, int32_t lmax,
                     float* out, void* workspace, size_t workspace_bytes,
                     zs_stream_t stream);

/*
 * zs_forward with coupling rows coup_ld floats apart (coup_ld >= D-1; row e
 * at coup + e * coup_ld, any 4-byte alignment): for instance the m = 0
 * segment of a packed Wigner band, read in place.  The banded storage of
 * the pull request "banded Wigner-D storage for the fused inference
 * consumers" keeps, per edge, three segments of the (E, 3*D-2) band, and
 * the GIE zonal coupling reads its m = 0 segment (section "What"); the
 * pages print no segment offsets, so the caller passes the pointer to the
 * first zonal row (the degree-1 entries after the degree-0 one) and the
 * band's row length, 3*D-2.  Results are bit-identical to zs_forward on the
 * same values stored contiguously.  Other arguments as zs_forward;
 * ZS_ERR_INVALID_ARG for coup_ld < D-1.
 */
ZS_API zs_status zs_forward_ld(const float* coup, int64_t coup_ld, const float* rad,
                               const int32_t* row_ptr, const int32_t* perm,
                               int64_t E, int32_t N, int32_t C, int32_t lmax,
                               float* out, void* workspace, size_t workspace_bytes, zs_stream_t stream);

/*
 * Forward with the degree normalisation fused in.  The pages apply an
 * inverse-square-root degree normalisation to the operator's output in the
 * traced graph, so that its own cotangent keeps flowing (pull request
 * "fused Triton zonal scatter for the GIE head", section "What", third
 * bullet, and its sequence diagram); here the per-node factor is applied
 * as the node is written, saving a pass over the (N, D, C) output.
 *   node_scale (N,)   per-node factor s[n] (for instance 1/sqrt of a
 *                     degree); any finite or non-finite value
 *   out (N, D, C)     out[n,1+r,c] = s[n] * (the zs_forward value), row 0
 *                     zero; nodes without edges are zero whatever s[n]
 *   out_raw (N, D, C) may be NULL; else also receives the unscaled
 *                     zs_forward result (what zs_backward_scaled needs for
 *                     the scale's gradient)
 * Other arguments, workspace, errors and summation order as zs_forward;
 * out equals zs_forward's result times s[n] rounded once (bitwise).
 */
ZS_API zs_status zs_forward_scaled(const float* coup, const float* rad,
                                   const int32_t* row_ptr, const int32_t* perm, const float* node_scale,
                                   int64_t E, int32_t N, int32_t C, int32_t lmax,
                                   float* out, float* out_raw, void* workspace, size_t workspace_bytes,
                                   zs_stream_t stream);

/*
 * Backward of zs_forward_scaled, edge order: for the cotangent g of the
 * scaled out,
 *   d_coup[e,r]  = s[dst[e]] * (zs_backward's d_coup with the same g)
 *   d_rad[e,l,c] = s[dst[e]] * (zs_backward's d_rad)
 *   d_scale[n]   = sum over rows 1..D-1 and channels of g[n,r,c] * out_raw[n,r,c]
 * node_scale (N,) as given to the forward; out_raw (N, D, C) the forward's
 * unscaled result, needed only when d_scale is not NULL; d_scale (N,) may
 * be NULL.  Each product of a gradient and s is rounded once.  Errors as
 * zs_backward, plus ZS_ERR_INVALID_ARG for a NULL node_scale, or a d_scale
 * without out_raw.  Needs no workspace.
 */
ZS_API zs_status zs_backward_scaled(const float* g, const float* coup, const float* rad, const int32_t* dst,
                                    const float* node_scale, const float* out_raw,
                                    int64_t E, int32_t N, int32_t C, int32_t lmax,
                                    float* d_coup, float* d_rad, float* d_scale, zs_stream_t stream);

/*
 * Backward of the zonal scatter (pull request "fused Triton zonal scatter
 * for the GIE head", section "What", backward bullet): one edge-parallel
 * pass writing both operand gradients.
 *   g (N,16,C)     cotangent of out; row 0 is not read
 *   coup, rad, dst the forward's inputs, indexed by edge id
 *   d_coup (E,15)  output, fully written
 *   d_rad (E,3,C)  output, fully written
 * Edges with dst outside [0, N) get zero gradients.  Needs no workspace.
 */
ZS_API zs_status zs_backward(const float* g, const float* coup, const float* rad,
                      const int32_t* dst, int64_t E, int32_t N, int32_t C, int32_t lmax,
                      float* d_coup, float* d_rad, zs_stream_t stream);

/*
 * zs_backward with coupling rows coup_ld floats apart and coupling-gradient
 * rows d_coup_ld floats apart (both >= D-1, any 4-byte alignment), so that
 * both can live in a packed band's m = 0 segment (see zs_forward_ld); only
 * the D-1 entries of each d_coup row are written.  Bit-identical to
 * zs_backward on contiguous copies.
 */
ZS_API zs_status zs_backward_ld(const float* g, const float* coup, int64_t coup_ld, const float* rad,
                                const int32_t* dst, int64_t E, int32_t N, int32_t C, int32_t lmax,
                                float* d_coup, int64_t d_coup_ld, float* d_rad, zs_stream_t stream);

/*
 * Backward of the zonal scatter with the edges visited in destination (CSR)
 * order: the same d_coup and d_rad as zs_backward, written for every edge,
 * for callers that already hold the forward's CSR.  Each node's cotangent
 * rows g[n] are read once per run of its edges instead of once per edge.
 *   g (N,16,C), coup (E,15), rad (E,3,C)  as for zs_backward
 *   row_ptr (N+1,), perm (E,)             the CSR zs_build_csr returned for
 *                                         the edges' destinations; perm must
 *                                         be a permutation of [0, E)
 *   d_coup (E,15), d_rad (E,3,C)          outputs, fully written; edges at
 *                                         positions >= row_ptr[N] (no node)
 *                                         get zero gradients
 * Needs no workspace.  Gradients agree with zs_backward's to fp32 rounding
 * (each is bitwise reproducible run to run).
 */
ZS_API zs_status zs_backward_csr(const float* g, const float* coup, const float* rad,
                                 const int32_t* row_ptr, const int32_t* perm,
                                 int64_t E, int32_t N, int32_t C, int32_t lmax,
                                 float* d_coup, float* d_rad, zs_stream_t stream);

/*
 * zs_forward without a workspace argument, for callers that cannot allocate
 * device memory: code that must not call cudaMalloc or a caching allocator
 * (for instance inside a region where allocation is forbidden or would
 * synchronise, or a host framework that owns all device memory and passes
 * in only the tensors).  The pages have no counterpart; this is a
 * convenience of this library.
 *   Arguments, results and errors as zs_forward (caller still passes the
 *   inputs and out).  The partial sums zs_forward keeps in its workspace
 *   live instead in one static device array of 4 MiB that every GPU
 *   loading the library holds until the process exits.  The single-kernel
 *   path (C == 32, rad 16-byte aligned, and out 16-byte aligned when
 *   lmax == 3; coup may have any 4-byte alignment) needs about 8 * R * 32
 *   bytes per SM whatever E is (R = (lmax+1)^2 - 1 rows, 3.8 KB at
 *   lmax 3); every other shape needs 8 * R * C + 12 bytes per 256 edges.
 *   A call that would need more returns ZS_ERR_INVALID_ARG and enqueues
 *   nothing.
 *   The first call on each device (and the first after a cudaDeviceReset)
 *   looks up the array's device address with cudaGetSymbolAddress, with
 *   that device current; make that first call before any stream capture.
 *   Every call shares the array: calls whose kernels overlap on the GPU
 *   (other streams, other host threads) race and give wrong results.
 *   Nothing in the array needs to start at zero.
 */
ZS_API zs_status zs_forward_noalloc(const float* coup, const float* rad,
                                    const int32_t* row_ptr, const int32_t* perm,
                                    int64_t E, int32_t N, int32_t C, int32_t lmax,
                                    float* out, zs_stream_t stream);

/*
 * Registers a caller-owned 32-bit word that the kernels set to 1 when a
 * bounded wait runs out (see zs_check_timeouts), so that a caller can see a
 * timeout without synchronising the device: for instance page-locked host
 * memory that the host reads at any time, or device memory that it copies
 * back asynchronously.  The word is only written (never cleared) by the
 * library; the caller clears it.
 *   flag   device memory, or page-locked host memory the device reaches at
 *          the same address (cudaHostAlloc / cudaMallocHost on a system
 *          with unified addressing), 4-byte aligned; NULL unregisters
 * Applies to the current device and to kernels enqueued after the call
 * (a synchronous copy to a device symbol: call it at set-up, not during
 * stream capture).  The word must stay valid until it is unregistered.
 * ZS_ERR_INVALID_ARG for memory the device cannot reach at that address.
 * The pages have no counterpart.
 */
ZS_API zs_status zs_set_timeout_flag(uint32_t* flag);

/*
 * Reads and clears the device-side count of bounded waits that ran out.
 * The kernels that stream operands with asynchronous bulk copies wait for
 * them with an iteration limit; a wait that reaches its limit is counted
 * and the kernel returns instead of hanging the GPU (its outputs are then
 * undefined), and the word registered with zs_set_timeout_flag, if any, is
 * set.  Synchronises the device.  Returns ZS_ERR_TIMEOUT when any
 * wait ran out since the previous call, ZS_OK otherwise.
 */
ZS_API zs_status zs_check_timeouts(void);

/*
 * Self-test of the bounded waits (the pages have no counterpart): enqueues a
 * one-warp kernel that waits on an mbarrier nothing completes, giving up
 * after max_spins tries (1 <= max_spins <= 2^16).  The wait records one
 * timeout, which the next
 * zs_check_timeouts() reports as ZS_ERR_TIMEOUT.  Nothing faults or hangs.
 */
ZS_API zs_status zs_selftest_bounded_wait(uint32_t max_spins, zs_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ZS_H_ */
