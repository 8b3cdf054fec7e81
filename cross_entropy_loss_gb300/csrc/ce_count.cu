// Count of the labels that take part in the mean: rows whose label is not
// ignore_index and lies in [0, V).  Under data parallelism every rank counts its
// own rows, the ranks sum the counts (one all-reduce of one integer), and each
// rank divides its share of the loss and gradient by that total -- the per-token
// mean across GPUs of the LossAccelerationPlugin (fms-hf-tuning PR #280, "Early
// Version Of This Plugin", `--loss_across_gpus mean token`).  The count is written
// as an int64 in device memory so the sum and its use by the fused kernel stay on
// the device, with no host round trip in between.
#include "common.cuh"
#include "foak_ce.h"
#include "internal.h"

namespace foak {

constexpr int kCountThreads = 1024;

__global__ void __launch_bounds__(kCountThreads) ce_count_valid_kernel(const int64_t* __restrict__ labels, int64_t N,
                                                                       int64_t V, int64_t ignore_index,
                                                                       int64_t* n_valid, int32_t* err) {
    griddep_launch_dependents();  // programmatic dependent launch: no global access before the wait
    griddep_wait();
    __shared__ int scratch[2 * (kCountThreads / 32)];
    int nv = 0, nb = 0;
    count_labels(labels, N, V, ignore_index, scratch, nv, nb);
    if (threadIdx.x == 0) {
        *n_valid = nv;
        if (err) *err = nb > 0 ? FOAK_ERRBIT_LABEL_RANGE : 0;
    }
}

cudaError_t launch_count_valid(const int64_t* labels, int64_t N, int64_t V, int64_t ignore_index, int64_t* n_valid,
                               int32_t* err, cudaStream_t stream) {
    return launch_dependent(ce_count_valid_kernel, dim3(1), dim3(kCountThreads), 0, stream, labels, N, V, ignore_index,
                            n_valid, err);
}

}  // namespace foak
