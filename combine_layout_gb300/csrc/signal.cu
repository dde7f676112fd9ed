// Device-side signals: a counter that producers add to when their data has
// landed, and a bounded wait that a consumer runs before reading that data.
//
// "NCCL EP 论文解读", item "设备API GIN": besides put and get, the device API
// offers SignalAdd (atomically add to a signal word) and WaitOnSignal (wait
// until the word reaches an expected value); item "send_only与双buffer": with
// send_only the send and the receive of a dispatch or combine are two
// kernels, and ncclEpComplete finishes the receive.  Here a send-only kernel's
// last CTA adds 1 to the handle's signal word after every CTA's stores
// (send_arrive, common.cuh), and moe_ep_complete enqueues the receive: one
// thread waits until the word holds the number of sends issued since the
// last completion, then takes that number off it, so the word is back at its
// starting value for the next micro-batch (also across CUDA-graph replays).
//
// The receive never runs concurrently with the sends it waits for: the host
// orders it after them (a stream-event join) before launching it, so in
// correct use its first poll succeeds.  Its wait is bounded in time and in
// polls; when the bound passes it latches the timeout slot of the group's
// device-error word and returns, leaving the word as it found it.
#include "common.cuh"

namespace moeep {
namespace {

constexpr uint32_t kMaxPolls = 1u << 26;  // polls before a wait gives up, whatever the clock says

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t load_acquire(const uint32_t* p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__global__ void __launch_bounds__(32) wait_signal_kernel(uint32_t* signal, uint32_t expected,
                                                         uint64_t limit_ns, unsigned* err)
{
    griddep_wait();
    if (threadIdx.x != 0) return;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 0; it < kMaxPolls; ++it) {
        if (load_acquire(signal) >= expected) {
            atomicSub(signal, expected);
            return;
        }
        if (global_ns() - t0 > limit_ns) break;
        __nanosleep(64);
    }
    *(volatile unsigned*)(err + kErrTimeout) = 1u;
}

__global__ void __launch_bounds__(32) signal_add_kernel(uint32_t* signal, uint32_t value)
{
    griddep_wait();
    if (threadIdx.x == 0)
        asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(signal), "r"(value)
                     : "memory");
}

}  // namespace

cudaError_t launch_wait_signal(uint32_t* signal, uint32_t expected, uint64_t limit_ns,
                               unsigned* err, cudaStream_t s)
{
    return launch_pdl(wait_signal_kernel, dim3(1), dim3(32), s, signal, expected, limit_ns, err);
}

cudaError_t launch_signal_add(uint32_t* signal, uint32_t value, cudaStream_t s)
{
    return launch_pdl(signal_add_kernel, dim3(1), dim3(32), s, signal, value);
}

}  // namespace moeep
