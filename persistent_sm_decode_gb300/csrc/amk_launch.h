/*
 * amk_launch.h — host-side entry points of the persistent kernel (defined in
 * amk_kernel.cu, used by amk_api.cpp).
 */
#pragma once
#include <cuda_runtime.h>

#include "amk_internal.h"

namespace amk {
typedef void (*KernelFn)(const Params);
/* kernel instance for the weight type (amk_weight_dtype) and the largest batch */
KernelFn select_kernel(int weight_dtype, int max_batch);
cudaError_t prepare_kernel(KernelFn fn, int smem_bytes);
cudaError_t occupancy(KernelFn fn, int smem_bytes, int *blocks_per_sm);
/* whether this build's kernel carries the per-task timing code (trace
 * option) and the loader's L2 prefetch (l2_prefetch_kb option) */
bool kernel_has_trace();
bool kernel_has_l2_prefetch();
/* one cooperative launch of n_sm CTAs */
cudaError_t launch_decode(KernelFn fn, const Params &p, int n_sm, int smem_bytes, cudaStream_t stream);
}  // namespace amk
