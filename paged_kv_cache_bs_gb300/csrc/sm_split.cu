// pa_sm_split: two disjoint SM partitions of one GPU, each with its own stream (CUDA green
// contexts).  A mixed chunked-prefill step holds a tensor-core-bound kernel (the prefill) and
// an HBM-bound one (the decode of the other sequences); the decode reaches the HBM bandwidth
// with well under half of the 152 SMs, so the two run side by side on disjoint SM sets
// instead of one after the other (pa_mixed_step).
//
// The green-context calls come from the driver entry points the runtime hands out, so the
// library still links against libcudart only.  Kernels are launched on the partition streams
// through the runtime API like any other stream.
#include <cuda.h>
#include <stdio.h>

#include <new>

#include "pa_common.cuh"

struct pa_sm_split {
    int device;
    int sms[2];
    CUgreenCtx ctx[2];
    cudaStream_t stream[2];
    cudaEvent_t fork;
    cudaEvent_t join[2];
};

namespace pa {
int set_last_error(int code, const char *msg);

namespace {

using DeviceGetFn = CUresult (*)(CUdevice *, int);
using GetDevResourceFn = CUresult (*)(CUdevice, CUdevResource *, CUdevResourceType);
using SplitByCountFn = CUresult (*)(CUdevResource *, unsigned int *, const CUdevResource *, CUdevResource *,
                                    unsigned int, unsigned int);
using GenerateDescFn = CUresult (*)(CUdevResourceDesc *, CUdevResource *, unsigned int);
using GreenCtxCreateFn = CUresult (*)(CUgreenCtx *, CUdevResourceDesc, CUdevice, unsigned int);
using GreenCtxDestroyFn = CUresult (*)(CUgreenCtx);
using GreenCtxStreamCreateFn = CUresult (*)(CUstream *, CUgreenCtx, unsigned int, int);
using StreamDestroyFn = CUresult (*)(CUstream);

struct Driver {
    DeviceGetFn device_get = nullptr;
    GetDevResourceFn get_resource = nullptr;
    SplitByCountFn split = nullptr;
    GenerateDescFn make_desc = nullptr;
    GreenCtxCreateFn ctx_create = nullptr;
    GreenCtxDestroyFn ctx_destroy = nullptr;
    GreenCtxStreamCreateFn stream_create = nullptr;
    StreamDestroyFn stream_destroy = nullptr;
    bool ok = false;
};

template <typename F>
bool entry(const char *name, F *fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12080, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
        return false;
    *fn = reinterpret_cast<F>(p);
    return true;
}

const Driver &driver() {
    static const Driver d = [] {
        Driver r;
        r.ok = entry("cuDeviceGet", &r.device_get) && entry("cuDeviceGetDevResource", &r.get_resource) &&
               entry("cuDevSmResourceSplitByCount", &r.split) && entry("cuDevResourceGenerateDesc", &r.make_desc) &&
               entry("cuGreenCtxCreate", &r.ctx_create) && entry("cuGreenCtxDestroy", &r.ctx_destroy) &&
               entry("cuGreenCtxStreamCreate", &r.stream_create) && entry("cuStreamDestroy", &r.stream_destroy);
        return r;
    }();
    return d;
}

int fail_cu(const char *what, CUresult r) {
    char msg[256];
    snprintf(msg, sizeof msg, "pa_sm_split_create: %s failed (CUresult %d)", what, static_cast<int>(r));
    return set_last_error(PA_ERR_CUDA, msg);
}

int fail_rt(const char *what, cudaError_t e) {
    char msg[256];
    snprintf(msg, sizeof msg, "%s: %s", what, cudaGetErrorString(e));
    return set_last_error(PA_ERR_CUDA, msg);
}

// Releases whatever part of the split exists (streams first, then their contexts).
void release(pa_sm_split *s) {
    const Driver &d = driver();
    for (int i = 0; i < 2; ++i) {
        if (s->join[i]) cudaEventDestroy(s->join[i]);
        if (s->stream[i]) {
            cudaStreamSynchronize(s->stream[i]);
            d.stream_destroy(static_cast<CUstream>(s->stream[i]));
        }
    }
    if (s->fork) cudaEventDestroy(s->fork);
    for (int i = 0; i < 2; ++i)
        if (s->ctx[i]) d.ctx_destroy(s->ctx[i]);
    delete s;
}

}  // namespace

cudaStream_t split_stream(const pa_sm_split *s, int i) { return s->stream[i]; }
int split_sms(const pa_sm_split *s, int i) { return s->sms[i]; }
int split_device(const pa_sm_split *s) { return s->device; }

cudaError_t split_fork(const pa_sm_split *s, cudaStream_t from) {
    cudaError_t e = cudaEventRecord(s->fork, from);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(s->stream[i], s->fork, 0);
    return e;
}

cudaError_t split_join(const pa_sm_split *s, cudaStream_t to) {
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
        e = cudaEventRecord(s->join[i], s->stream[i]);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(to, s->join[i], 0);
    }
    return e;
}

}  // namespace pa

extern "C" {

PA_API int pa_sm_split_create(int32_t first_sms, pa_sm_split **out) {
    using pa::set_last_error;
    if (!out) return set_last_error(PA_ERR_INVALID_ARG, "pa_sm_split_create: out is NULL");
    *out = nullptr;
    const pa::Driver &d = pa::driver();
    if (!d.ok) return set_last_error(PA_ERR_UNSUPPORTED, "pa_sm_split_create: the driver has no green-context calls");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaSetDevice(dev);  // the primary context exists before the partitions
    if (e != cudaSuccess) return pa::fail_rt("pa_sm_split_create", e);
    CUdevice cdev;
    CUresult r = d.device_get(&cdev, dev);
    if (r != CUDA_SUCCESS) return pa::fail_cu("cuDeviceGet", r);
    CUdevResource all = {};
    r = d.get_resource(cdev, &all, CU_DEV_RESOURCE_TYPE_SM);
    if (r != CUDA_SUCCESS) return pa::fail_cu("cuDeviceGetDevResource", r);
    const int total = static_cast<int>(all.sm.smCount);
    const int align = all.sm.smCoscheduledAlignment > 0 ? static_cast<int>(all.sm.smCoscheduledAlignment) : 1;
    const int min_part = static_cast<int>(all.sm.minSmPartitionSize);
    if (first_sms <= 0 || first_sms % align || first_sms < min_part || total - first_sms < min_part) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "pa_sm_split_create: first_sms %d must be a multiple of %d, at least %d, and leave at least %d of "
                 "the device's %d SMs",
                 first_sms, align, min_part, min_part, total);
        return set_last_error(PA_ERR_INVALID_ARG, msg);
    }
    CUdevResource part[1] = {}, rest = {};
    unsigned int groups = 1;
    r = d.split(part, &groups, &all, &rest, 0, static_cast<unsigned int>(first_sms));
    if (r != CUDA_SUCCESS) return pa::fail_cu("cuDevSmResourceSplitByCount", r);
    if (groups != 1 || static_cast<int>(part[0].sm.smCount) != first_sms)
        return set_last_error(PA_ERR_UNSUPPORTED, "pa_sm_split_create: the driver did not make the partition asked for");

    pa_sm_split *s = new (std::nothrow) pa_sm_split{};
    if (!s) return set_last_error(PA_ERR_CUDA, "pa_sm_split_create: out of host memory");
    s->device = dev;
    CUdevResource *res[2] = {&part[0], &rest};
    for (int i = 0; i < 2; ++i) {
        CUdevResourceDesc desc;
        r = d.make_desc(&desc, res[i], 1);
        if (r == CUDA_SUCCESS) r = d.ctx_create(&s->ctx[i], desc, cdev, CU_GREEN_CTX_DEFAULT_STREAM);
        CUstream st = nullptr;
        if (r == CUDA_SUCCESS) r = d.stream_create(&st, s->ctx[i], CU_STREAM_NON_BLOCKING, 0);
        if (r != CUDA_SUCCESS) {
            pa::release(s);
            return pa::fail_cu("creating a green context and its stream", r);
        }
        s->stream[i] = static_cast<cudaStream_t>(st);
        s->sms[i] = static_cast<int>(res[i]->sm.smCount);
    }
    e = cudaEventCreateWithFlags(&s->fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s->join[0], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s->join[1], cudaEventDisableTiming);
    if (e != cudaSuccess) {
        pa::release(s);
        return pa::fail_rt("pa_sm_split_create: cudaEventCreateWithFlags", e);
    }
    *out = s;
    pa::set_last_error(PA_OK, "");
    return PA_OK;
}

PA_API int pa_sm_split_info(const pa_sm_split *split, int32_t *first_sms, int32_t *second_sms, void **first_stream,
                            void **second_stream) {
    if (!split) return pa::set_last_error(PA_ERR_INVALID_ARG, "pa_sm_split_info: split is NULL");
    if (first_sms) *first_sms = split->sms[0];
    if (second_sms) *second_sms = split->sms[1];
    if (first_stream) *first_stream = split->stream[0];
    if (second_stream) *second_stream = split->stream[1];
    return PA_OK;
}

PA_API void pa_sm_split_destroy(pa_sm_split *split) {
    if (split) pa::release(split);
}

}  // extern "C"
