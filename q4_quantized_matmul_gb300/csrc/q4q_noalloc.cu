// q4q_noalloc.cu -- q4q_mul_mat for callers that cannot allocate device memory.
//
// Some callers have no way to hand this library scratch memory: a plugin inside
// a host application whose allocator owns every byte of device memory (an
// inference server with its own memory pool, a runtime that forbids allocation
// once it has started), or a C caller that only ever receives the input and
// output pointers.  For them this file keeps the scratch space of the
// tensor-core path (and of the generic path) in one statically sized device
// array that the library owns, so the call needs nothing but inputs and outputs.
//
// The array lives in every GPU that loads the library, for the life of the
// process.  Its device address is looked up once per device, on the first call
// made while that device is current (cudaGetSymbolAddress), and cached.
#include <mutex>

#include "q4q_common.cuh"
#include "q4q_internal.h"

namespace q4q {
namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = Q4Q_NOALLOC_SCRATCH_BYTES;   // 8 MiB per device

static __device__ __align__(256) uint8_t g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[MAX_DEVICES] = {};

// Device address of the static scratch array on the current device.  The host
// symbol g_noalloc_scratch is only a stand-in for it and must never reach a kernel.
q4q_status scratch_address(int device, void** out) {
    if (device < 0 || device >= MAX_DEVICES) return Q4Q_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[device]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return Q4Q_ERR_CUDA;
        g_scratch_ptr[device] = p;
    }
    *out = g_scratch_ptr[device];
    return Q4Q_OK;
}

}  // namespace
}  // namespace q4q

extern "C" q4q_status q4q_mul_mat_noalloc(const void* src0, int64_t ne00, int64_t ne01,
                                          const float* src1, int64_t ne10, int64_t ne11,
                                          float* dst, q4q_stream_t stream) {
    size_t need = 0;
    q4q_status st = q4q::mul_mat_min_workspace_bytes(ne00, ne01, ne11, &need);
    if (st != Q4Q_OK) return st;
    if (ne10 != ne00) return Q4Q_ERR_SHAPE;
    if (ne01 == 0 || ne11 == 0) return Q4Q_OK;
    if (need > q4q::NOALLOC_SCRATCH_BYTES) return Q4Q_ERR_WORKSPACE;
    q4q::DeviceInfo info;
    if ((st = q4q::current_device_info(&info)) != Q4Q_OK) return st;
    void* scratch = nullptr;
    if ((st = q4q::scratch_address(info.device, &scratch)) != Q4Q_OK) return st;
    return q4q_mul_mat(src0, ne00, ne01, src1, ne10, ne11, dst, scratch, q4q::NOALLOC_SCRATCH_BYTES, stream);
}
