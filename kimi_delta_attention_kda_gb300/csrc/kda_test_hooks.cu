// kda_test_hooks.cu -- test-only entry points that make the library's bounded
// waits run out, so that their exit path is exercised on the GPU.
//
// Compiled only into the test library libkda_testhooks.so, with
// KDA_TEST_HOOKS defined and KDA_WAIT_BOUND_CYCLES = 10^5 (about 50 us), never
// into libkda.so.  Each hook launches one CTA that uses the waits of the real
// kernels (kda_common.cuh) on a ring nobody completes or a ready flag nobody
// sets.  A wait that runs out sets kDevPipeTimeout and returns; the kernel
// then leaves with nothing in flight, and the context stays usable.  Nothing
// here faults or hangs: every wait is bounded, every copy stays inside the
// caller's buffer and the CTA's shared memory.
#ifdef KDA_TEST_HOOKS
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kRingStages = 4;
constexpr uint32_t kRingStageBytes = 1024;

// One producer warp (warp 2) and two consumer warps (0, 1) on a ring of four
// stages, as in the recurrence kernels: the producer fills `filled` stages
// (0 .. filled-1, one bulk copy of 1 KB each from src) and never fills the
// next one; the consumers take the stages in order with the warp-uniform
// bounded wait and stop at the first wait that runs out.  out[0] = chunks
// the consumers saw, out[1] = 1 if the consumers' wait ran out.
__global__ void __launch_bounds__(96, 1)
    stalled_ring_kernel(const uint8_t* src, int filled, int* status, int* out) {
    __shared__ __align__(128) uint8_t ring[kRingStages][kRingStageBytes];
    __shared__ uint64_t full[kRingStages];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRingStages; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (warp == 2) {
        if (lane == 0)
            for (int s = 0; s < filled && s < kRingStages - 1; ++s) {
                mbar_arrive_expect_tx(&full[s], kRingStageBytes);
                bulk_g2s(ring[s], src + s * kRingStageBytes, kRingStageBytes, &full[s]);
            }
        __syncwarp();
        return;   // the next stage is never filled
    }
    int seen = 0;
    bool ok = true;
    for (int s = 0; s < kRingStages && ok; ++s) {
        ok = mbar_wait_warp(&full[s], 0, status);
        if (ok) ++seen;
    }
    if (threadIdx.x == 0) {
        out[0] = seen;
        out[1] = ok ? 0 : 1;
    }
}

// One warp waits for ready flags[0] (stride 1, 32 at a time) with the poll of
// the one-launch form; nothing ever sets it.  out[2] = 1 if the wait ran out.
__global__ void unset_flag_kernel(const uint32_t* flags, int* status, int* out) {
    uint32_t mask = 0;
    const bool ok = wait_ready_flags(flags, 1, 32, &mask, status);
    if (threadIdx.x == 0) out[2] = ok ? 0 : 1;
}

}  // namespace
}  // namespace kda

using namespace kda;

// The two hooks on `stream`: src a device buffer of at least 3 KB (16-byte
// aligned), flags 32 zero uint32 flags, status and out device ints
// (status: KDA_DEV_* bits ORed in; out: 3 ints).  Returns a cudaError_t.
extern "C" int kda_test_wait_bounds(const void* src, const uint32_t* flags, int* status,
                                    int* out, void* stream_ptr) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    stalled_ring_kernel<<<1, 96, 0, stream>>>(static_cast<const uint8_t*>(src), 3, status, out);
    unset_flag_kernel<<<1, 32, 0, stream>>>(flags, status, out);
    return static_cast<int>(cudaGetLastError());
}

// The wait bound this library was compiled with, in clock cycles.
extern "C" long long kda_test_wait_bound_cycles(void) { return kWaitBoundCycles; }
#endif  // KDA_TEST_HOOKS
