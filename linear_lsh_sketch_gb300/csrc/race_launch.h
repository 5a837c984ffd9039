// race_launch.h -- host-side launchers of the RACE attention kernels (internal to the library).
#pragma once

#include <algorithm>

#include "race_common.cuh"

namespace race {

// Instrumentation hooks implemented next to the C ABI: a launch counter and optional CUDA
// event pairs around each launch.
void prof_before(const char *name, cudaStream_t st);
void prof_after(const char *name, cudaStream_t st);

template <typename Kern, typename... Args>
cudaError_t launch_kernel(const char *name, Kern k, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                          Args... args)
{
    prof_before(name, st);
    k<<<grid, block, smem, st>>>(args...);
    cudaError_t e = cudaGetLastError();
    prof_after(name, st);
    return e;
}

// Streaming multiprocessors of the current device (152 when no device can be queried).
int device_sm_count();

// ---------------------------------------------------------------- causal decode step
bool decode_supported(const Dims &D);
template <typename T>
cudaError_t launch_decode(const Dims &D, const T *q, const T *k, const T *v, const float *W, float *S, T *o,
                          cudaStream_t st);

// ---------------------------------------------------------------- exact angular attention
template <typename T>
cudaError_t launch_angular(const Dims &D, const T *Q, const T *K, const T *V, float gamma, int causal, T *O,
                           cudaStream_t st);

// ---------------------------------------------------------------- CUDA-core kernels
enum class GenericKernel { Sketch, Readout, QueryBwd, KeyBwd, CausalFwd, CausalBwd };
size_t generic_smem_bytes(const Dims &D, GenericKernel which);
int generic_token_tile();

template <typename T>
cudaError_t launch_sketch(const Dims &D, const T *X, const T *Y, const float2 *aux, const float *W,
                          int64_t seg_len, int nsplit, float *part, int mode, cudaStream_t st);
cudaError_t launch_combine(const Dims &D, const float *part, float *out, int nsplit, int mode, cudaStream_t st);
// dbeta[bh] from the backward kernels' d(loss)/d(beta) partials, two [BH][slots] float arrays.
cudaError_t launch_dbeta_combine(const Dims &D, const float *part, int slots, float *dbeta, cudaStream_t st);
// d(loss)/d(W) per (b, h), [BH][L P][d], from the dz / |x| rows in D.dzq and D.dzk: nblk token
// ranges per (b, h) write partials [BH][nblk][L P][d] to part, then a fixed-order sum.
template <typename T>
cudaError_t launch_dw(const Dims &D, const T *Q, const T *K, int nblk, float *part, float *dW, cudaStream_t st);
template <typename T>
cudaError_t launch_readout(const Dims &D, const T *Q, const float *W, const float *S, T *O, unsigned *err,
                           cudaStream_t st);
template <typename T>
cudaError_t launch_bwd_query(const Dims &D, const T *Q, const T *dO, const float *W, const float *S, T *dQ,
                             float2 *aux, float *dbpart, cudaStream_t st);
template <typename T>
cudaError_t launch_bwd_key(const Dims &D, const T *K, const T *V, const float *W, const float *G, T *dK, T *dV,
                           float *dbpart, cudaStream_t st);
template <typename T>
cudaError_t launch_causal_fwd(const Dims &D, const T *Q, const T *K, const T *V, const float *W, const float *S0,
                              int64_t seg_len, int nseg, T *O, unsigned *err, cudaStream_t st);
template <typename T>
cudaError_t launch_causal_bwd_q(const Dims &D, const T *Q, const T *K, const T *V, const T *dO, const float *W,
                                const float *S0, int64_t seg_len, int nseg, T *dQ, float2 *aux, float *dbpart,
                                cudaStream_t st);
template <typename T>
cudaError_t launch_causal_bwd_kv(const Dims &D, const T *Q, const T *K, const T *V, const T *dO,
                                 const float2 *aux, const float *W, const float *G0, int64_t seg_len, int nseg,
                                 T *dK, T *dV, float *dbpart, cudaStream_t st);

// ---------------------------------------------------------------- tcgen05 non-causal path (bf16)
bool nc5_supported(const Dims &D);
int nc5_tile();
int nc5_sketch_ctas_per_sm(const Dims &D);
// frows, invrows (optional, together): also every token's bucket-feature row of X, bf16
// [BH][N][feature row stride], and its 1 / |x|, fp32 [BH][N].
cudaError_t launch_nc5_sketch(const Dims &D, const bf16_t *X, const bf16_t *Y, const float2 *aux, const float *W,
                              int64_t seg_len, int nsplit, float *part, unsigned *err, cudaStream_t st,
                              bf16_t *frows = nullptr, float *invrows = nullptr);
cudaError_t launch_nc5_readout(const Dims &D, const bf16_t *Q, const float *W, const float *S, bf16_t *O,
                               unsigned *err, cudaStream_t st);
bool c5_supported(const Dims &D);
// fk: every key's bucket-feature row, bf16 [BH][N][feature row stride], as the segment-sum pass
// (launch_nc5_sketch with frows) stores it.
cudaError_t launch_c5_fwd(const Dims &D, const bf16_t *Q, const bf16_t *fk, const bf16_t *V, const float *W,
                          const float *S0, int64_t seg_len, int nseg, bf16_t *O, unsigned *err, cudaStream_t st);
bool c5_bwd_supported(const Dims &D);
// Bytes of one [BH][N][feature row stride] bf16 array of bucket-feature rows.  The query-side
// pass reads the keys' rows fk (as the forward's segment-sum pass stored them) in place of K, and
// writes F'_Q = phi(Q_t) / den_t (fq), which the key-side pass reads in place of Q.
size_t c5_feature_rows_bytes(const Dims &D);
cudaError_t launch_c5_bwd_q(const Dims &D, const bf16_t *Q, const bf16_t *fk, const bf16_t *V, const bf16_t *dO,
                            const float *W, const float *S0, int64_t seg_len, int nseg, bf16_t *dQ, float2 *aux,
                            bf16_t *fq, float *Gseg, unsigned *err, float *dbpart, cudaStream_t st);
// The key-side pass also reads the keys' feature rows fk and their 1 / |k| (kinv), as the
// forward's segment-sum pass stored them, instead of normalising and featurising K again.
cudaError_t launch_c5_bwd_kv(const Dims &D, const bf16_t *fq, const bf16_t *fk, const float *kinv, const bf16_t *K,
                             const bf16_t *V, const bf16_t *dO, const float2 *aux, const float *W, const float *G0,
                             int64_t seg_len, int nseg, bf16_t *dK, bf16_t *dV, unsigned *err, float *dbpart,
                             cudaStream_t st);
// Token segments per (b, h) of the two non-causal tcgen05 backward kernels (their grid's x).
int nc5_bwd_nseg(const Dims &D);
cudaError_t launch_nc5_bwd_query(const Dims &D, const bf16_t *Q, const bf16_t *dO, const float *W, const float *S,
                                 bf16_t *dQ, float2 *aux, unsigned *err, float *dbpart, cudaStream_t st);
cudaError_t launch_nc5_bwd_key(const Dims &D, const bf16_t *K, const bf16_t *V, const float *W, const float *G,
                               bf16_t *dK, bf16_t *dV, unsigned *err, float *dbpart, cudaStream_t st);

}  // namespace race
