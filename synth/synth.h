/*
 * synth.h - seeded synthetic inputs for the lockstep tick (test and bench infrastructure).
 *
 * This module generates the random-init weights, ring-KV contents and token streams
 * that stand in for trained PersonaPlex checkpoints, voice prompts and Mimi codes,
 * none of which exist here.  It holds none of the tick's arithmetic: it only turns
 * (seed, stream, index) into numbers.  Both the CPU oracle's callers and the CUDA
 * path's callers use it, so the two sides see bit-identical inputs without sharing
 * any code with each other.
 *
 * Generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers:
 * as easy as 1, 2, 3", SC 2011), counter = (index lo, index hi, stream, 0),
 * key = (seed, 0).  Each 128-bit output gives eight 16-bit uniforms u_0..u_7
 * (word w, low half first).  A normal deviate is the centred 8-term Irwin-Hall
 * sum: the integer S = u_0 + ... + u_7 - 262140 (262140 = 8 * 65535 / 2, so the
 * mean is exactly zero), converted exactly to fp32, times an fp32 scale
 * c = sigma / sd(S) (one rounding), then rounded to bf16 to nearest-even.  Every step is integer or a single IEEE fp32 multiply, so
 * the host (C) and device (CUDA) implementations agree bit for bit.
 */
#ifndef PP_SYNTH_H
#define PP_SYNTH_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* One Philox4x32-10 block: ctr[4], key[2] -> out[4]. */
void ppsyn_philox(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* fp32 scale that maps the centred 8-term Irwin-Hall sum to standard deviation sigma. */
float ppsyn_normal_scale(double sigma);

/* out[i] = bf16(normal(seed, stream, i0 + i) * sigma) for i < n (host, OpenMP). */
void ppsyn_normal_bf16_host(uint16_t* out, int64_t n, int64_t i0, uint32_t seed,
                            uint32_t stream, float scale);

/* out[i] = fp32 deviate before the bf16 rounding (host), for distribution checks. */
void ppsyn_normal_f32_host(float* out, int64_t n, int64_t i0, uint32_t seed,
                           uint32_t stream, float scale);

/* out[i] = lo + floor(u32 * (hi - lo) / 2^32), u32 = word 0 of block (seed, stream, i0+i). */
void ppsyn_uniform_i32_host(int32_t* out, int64_t n, int64_t i0, uint32_t seed,
                            uint32_t stream, int32_t lo, int32_t hi);

/* Device twin of ppsyn_normal_bf16_host; out is a device pointer; returns a cudaError_t. */
int ppsyn_normal_bf16_dev(uint16_t* out, int64_t n, int64_t i0, uint32_t seed,
                          uint32_t stream, float scale, void* cuda_stream);

/* Device fill of a strided set of contiguous blocks: block j (0 <= j < nblk) of
 * blk_elems elements starts at out + j*blk_stride and takes indices
 * i0 + j*blk_elems ...  Used to fill one slot's ring across all layers. */
int ppsyn_normal_bf16_dev_blocks(uint16_t* out, int64_t nblk, int64_t blk_elems,
                                 int64_t blk_stride, int64_t i0, uint32_t seed,
                                 uint32_t stream, float scale, void* cuda_stream);

#ifdef __cplusplus
}
#endif
#endif
