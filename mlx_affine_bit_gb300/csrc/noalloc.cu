// noalloc.cu -- tf_qmm_noalloc: the product with no device allocation at all.
//
// Some callers cannot let a library call cudaMalloc: code that runs while a
// stream is being captured into a CUDA graph, engines that hand all device
// memory to their own pool up front, and processes that must not grow their
// device footprint after start-up.  tf_qmm allocates a split-K workspace and a
// status word on first use; this entry point instead takes that scratch from
// one fixed array compiled into the library.
//
// The array holds, in order, a status word, the split-K arrival counters and
// the split-K partial sums.  Every GPU that loads the library holds it until
// the process exits.  Every call shares it and it keeps the last call's
// contents, so each call clears the counters it uses on its own stream first;
// calls that overlap on the GPU (for example on two streams at once) race on
// it.  The status word is cleared once at set-up and then only by
// tf_noalloc_status, so a bounded wait that ran out stays recorded until the
// caller reads it.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/tfqmm.h"
#include "internal.h"

namespace {

constexpr size_t SCRATCH_BYTES = 4u << 20;        // the fixed maximum: 4 MiB per device
constexpr size_t STATUS_BYTES = 256;
constexpr size_t COUNTER_BYTES = 64u << 10;       // arrival counters: up to 16384 column tiles
constexpr size_t PARTIAL_BYTES = SCRATCH_BYTES - STATUS_BYTES - COUNTER_BYTES;
constexpr int MAX_DEVICES = 64;

static __device__ __align__(256) unsigned char scratch[SCRATCH_BYTES];

struct DeviceScratch {
    unsigned char *base = nullptr;   // device address of `scratch` on this device
    int nsm = 0;
};

std::mutex g_mu;
DeviceScratch g_dev[MAX_DEVICES];

// Once per device, with that device current: the array's device address (the
// host-side name `scratch` is only a stand-in, never a device address).
int device_scratch(DeviceScratch **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return tfq::fail_message(TF_ECUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= MAX_DEVICES) return tfq::fail_message(TF_EINVAL_SIZE, "device ordinal out of range");
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceScratch &d = g_dev[dev];
    if (!d.base) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, scratch);
        if (e != cudaSuccess || !ptr)
            return tfq::fail_message(TF_ECUDA, "cudaGetSymbolAddress(scratch) failed");
        e = cudaDeviceGetAttribute(&d.nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return tfq::fail_message(TF_ECUDA, "cudaDeviceGetAttribute failed");
        e = cudaMemset(ptr, 0, STATUS_BYTES);
        if (e != cudaSuccess) return tfq::fail_message(TF_ECUDA, "cudaMemset(scratch status) failed");
        d.base = static_cast<unsigned char *>(ptr);
    }
    *out = &d;
    return TF_OK;
}

}  // namespace

extern "C" int tf_qmm_noalloc(const uint16_t *x, int rows, int K, const uint32_t *W,
                              const uint16_t *scales, const uint16_t *biases, int N, int bits,
                              int group, float *y, int64_t y_stride, void *stream) {
    DeviceScratch *d = nullptr;
    const int rc = device_scratch(&d);
    if (rc) return rc;
    int *status = reinterpret_cast<int *>(d->base);
    int *counters = reinterpret_cast<int *>(d->base + STATUS_BYTES);
    float *partials = reinterpret_cast<float *>(d->base + STATUS_BYTES + COUNTER_BYTES);
    return tfq::product_with_scratch(x, rows, K, W, scales, biases, N, bits, group, y, y_stride,
                                     static_cast<cudaStream_t>(stream), d->nsm, partials,
                                     PARTIAL_BYTES / sizeof(float), counters,
                                     COUNTER_BYTES / sizeof(int), status);
}

extern "C" int tf_noalloc_status(void) {
    DeviceScratch *d = nullptr;
    const int rc = device_scratch(&d);
    if (rc) return rc;
    int v = 0;
    cudaError_t e = cudaMemcpy(&v, d->base, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return tfq::fail_message(TF_ECUDA, "cudaMemcpy(scratch status) failed");
    if (v) {
        e = cudaMemset(d->base, 0, sizeof v);
        if (e != cudaSuccess) return tfq::fail_message(TF_ECUDA, "cudaMemset(scratch status) failed");
        if (v & tfq::STATUS_BOUNDS)
            return tfq::fail_message(TF_EBOUNDS, "the debug build found an index outside its buffer");
        return tfq::fail_message(TF_EDEVICE, "a no-allocation product gave up a bounded wait");
    }
    return tfq::fail_message(TF_OK, "");
}
