// debug.cu - sentinel checks of the receive buffer (EP_DEBUG=1, read at
// ep_buffer_init). The dispatch fills the call's receive rows with 0xFF
// before its permute; this kernel then checks every row: a row inside its
// rank's true total must have been written (its first 16 bytes are not all
// 0xFF, which no finite input row produces), and a row past it must still
// hold the sentinel (nothing wrote outside the layout). The combine runs the
// same check when it reads the receive buffer itself. Violations set
// kErrDebugUnwritten / kErrDebugStray in the device error word; nothing traps.
#include "ep_device.cuh"
#include "ep_next.cuh"

namespace ep {
namespace {

constexpr int kCheckThreads = 256;

__global__ void __launch_bounds__(kCheckThreads)
sentinel_check_kernel(SentinelArgs a)
{
    griddep_wait();
    const int64_t rows = (int64_t)a.R * a.S;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int32_t total = __ldcg(a.rank_prefix + a.R - 1);
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < rows; q += stride) {
        bool valid;
        if (a.packed) {
            valid = q < total;
        } else {
            const int64_t r = q / a.S;
            valid = (q - r * a.S) < __ldcg(a.rows_per_rank + r);
        }
        const int4 v = ld_cg_v4(reinterpret_cast<const int4*>(a.recv_x + q * a.row_bytes));
        const bool sentinel = (v.x & v.y & v.z & v.w) == -1;
        if (valid && sentinel) atomicOr(a.err, kErrDebugUnwritten);
        if (!valid && !sentinel) atomicOr(a.err, kErrDebugStray);
    }
    griddep_launch_dependents();
}

}  // namespace

cudaError_t launch_sentinel_check(const SentinelArgs& a, int num_sms, const LaunchOpts& o)
{
    const int64_t rows = (int64_t)a.R * a.S;
    if (rows <= 0) return cudaSuccess;
    int64_t grid = (rows + kCheckThreads - 1) / kCheckThreads;
    const int64_t cap = (int64_t)(num_sms > 0 ? num_sms : 1) * 8;
    if (grid > cap) grid = cap;
    return launch_kernel(sentinel_check_kernel, dim3((unsigned)grid), dim3(kCheckThreads), 0, o, a);
}

}  // namespace ep
