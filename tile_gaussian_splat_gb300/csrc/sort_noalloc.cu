// gs_sort_pairs_noalloc: the stable pair sort of gs_sort_pairs for callers
// that cannot allocate device memory -- code that runs inside a host
// framework which owns every device allocation and forbids others, or a
// loop that must never pay for an allocation -- and so cannot supply the
// workspace gs_sort_pairs asks for.
//
// The scratch space (digit histograms, look-back words, block tickets, the
// error flag and the alternate key/value buffers) is a file-scope device
// array of fixed size, sized for at most kNoAllocMaxPairs pairs.  Every GPU
// that loads this library holds one copy of it until the process exits.
// The array's name in host code is only a host-side stand-in, so the device
// address is fetched with cudaGetSymbolAddress, once per device, with that
// device current, and passed to the kernels.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/gs_splat.h"
#include "gs_internal.h"

namespace {

using namespace gs;

constexpr int64_t kNoAllocMaxPairs = GS_SORT_NOALLOC_MAX_PAIRS;
constexpr int kPasses = 8;
constexpr size_t kAlignBytes = 256;

constexpr size_t round_up(size_t v) { return (v + kAlignBytes - 1) / kAlignBytes * kAlignBytes; }

constexpr size_t kBlocks = (size_t)((kNoAllocMaxPairs + kTile64 - 1) / kTile64);
constexpr size_t kOffTickets = round_up(sizeof(int32_t));                       // after the error flag
constexpr size_t kOffHist = kOffTickets + round_up(kPasses * sizeof(uint32_t));
constexpr size_t kOffLookback = kOffHist + round_up(kPasses * 256 * sizeof(uint32_t));
// look-back words: a call over n pairs uses passes * sort_blocks(n) * 256 of
// them, packed from kOffLookback (a pass's region starts right after the
// previous pass's), so only that much needs clearing per call
constexpr size_t kLookbackBytes = kPasses * kBlocks * 256 * sizeof(uint64_t);
constexpr size_t kOffAltKeys = round_up(kOffLookback + kLookbackBytes);
constexpr size_t kOffAltVals = kOffAltKeys + round_up(kNoAllocMaxPairs * sizeof(uint64_t));
constexpr size_t kScratchBytes = kOffAltVals + round_up(kNoAllocMaxPairs * sizeof(int32_t));

// 20,980,224 bytes (about 21.0 MB) per device: 8 passes x 512 blocks x 256
// look-back words x 8 bytes, 8 MB of alternate keys, 4 MB of alternate
// values and 8.7 KB of flag, tickets and histograms.
static_assert(kScratchBytes == 20980224, "the stated size of the scratch array");
static __device__ __align__(256) unsigned char g_sort_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned char* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_sort_scratch on the current device (fetched once).
int scratch_for_current_device(unsigned char** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GS_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GS_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_sort_scratch) != cudaSuccess || !p) return GS_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
    }
    *out = g_scratch_ptr[dev];
    return GS_OK;
}

}  // namespace

extern "C" int gs_sort_pairs_noalloc(uint64_t* keys, int32_t* values, int64_t n, int begin_bit,
                                     int end_bit, int32_t* d_status, void* stream) {
    if (n < 0 || begin_bit < 0 || end_bit > 64 || begin_bit > end_bit ||
        (n > 0 && (!keys || !values)))
        return GS_ERR_INVALID_ARG;
    if (n > kNoAllocMaxPairs) return GS_ERR_CAPACITY;
    if (n <= 1 || begin_bit == end_bit) return GS_OK;
    unsigned char* base = nullptr;
    const int rc = scratch_for_current_device(&base);
    if (rc != GS_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t* abort_flag = reinterpret_cast<int32_t*>(base);
    uint32_t* tickets = reinterpret_cast<uint32_t*>(base + kOffTickets);
    uint32_t* hist = reinterpret_cast<uint32_t*>(base + kOffHist);
    uint64_t* alt_k = reinterpret_cast<uint64_t*>(base + kOffAltKeys);
    int32_t* alt_v = reinterpret_cast<int32_t*>(base + kOffAltVals);
    // the array keeps the previous call's contents: clear the flag, tickets,
    // histograms and the look-back words of this call's passes, which must
    // start at zero
    const int passes = (end_bit - begin_bit + 7) / 8;
    const size_t lb_words = (size_t)sort_blocks(n, kTile64) * 256;
    const size_t zero_bytes = kOffLookback + (size_t)passes * lb_words * sizeof(uint64_t);
    if (cudaMemsetAsync(base, 0, zero_bytes, s) != cudaSuccess) return GS_ERR_CUDA;
    launch_digit_hist_u64(keys, n, begin_bit, end_bit, hist, s);
    uint64_t* sk = keys;
    int32_t* sv = values;
    for (int pass = 0; pass < passes; ++pass) {
        uint64_t* dk = sk == keys ? alt_k : keys;
        int32_t* dv = sv == values ? alt_v : values;
        uint64_t* lb = reinterpret_cast<uint64_t*>(base + kOffLookback) + (size_t)pass * lb_words;
        launch_onesweep_u64(sk, sv, dk, dv, n, begin_bit + 8 * pass, end_bit, hist + 256 * pass,
                            LookbackScratch{lb, tickets + pass}, abort_flag, d_status, s);
        sk = dk;
        sv = dv;
    }
    if (sk != keys) {
        if (cudaMemcpyAsync(keys, sk, (size_t)n * 8, cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
            cudaMemcpyAsync(values, sv, (size_t)n * 4, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return GS_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? GS_OK : GS_ERR_CUDA;
}
