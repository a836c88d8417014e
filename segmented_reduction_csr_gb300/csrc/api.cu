// api.cu -- the C ABI of libsegreduce (declared in include/seg_reduce.h):
// argument checks, the host launch planner, the library-owned scratch cache
// and the kernel launch.  Nothing here reads device memory on the host.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/seg_reduce.h"
#include "seg_pick.cuh"
#include "seg_plan.cuh"
#include "seg_rle.cuh"
#include "seg_scan.cuh"
#include "seg_scatter.cuh"
#include "seg_seq.cuh"
#include "seg_sort.cuh"

using namespace segred;

namespace {

constexpr int32_t kVersion = 1 * 10000 + 0 * 100 + 0;
constexpr int kMaxDevices = 64;

// Self-test of the bounded waits: one thread waits, with the kernels' own
// wait_bounded_for, on an mbarrier phase that nothing completes; the wait
// runs out after limit_ns, ORs STATUS_CONSUMER_TIMEOUT into the status word
// and the kernel returns.  No copy is in flight and nothing else waits.
__global__ void selftest_wait_kernel(unsigned int* status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    mbar_init(&bar, 1);
    fence_mbarrier_init();
    (void)wait_bounded_for(&bar, 0, status, STATUS_CONSUMER_TIMEOUT, limit_ns);
}

// ---------------------------------------------------------------------------
// Per-device state: SM count, status word, kernels already configured.

struct DeviceState {
    bool init = false;
    int sm_count = 0;
    unsigned int* status = nullptr;
    std::map<const void*, bool> configured;
};

struct Scratch {
    void* ptr = nullptr;
    size_t bytes = 0;
    uint32_t gen = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::map<std::pair<int, cudaStream_t>, Scratch> g_scratch;
// The deterministic scatter's sort buffers, offsets and gathered rows: a
// buffer of their own per (device, stream), so that the reduction it runs
// keeps its scratch (and its ticket words) to itself.
std::map<std::pair<int, cudaStream_t>, Scratch> g_sort_scratch;

seg_status_t device_state(int dev, DeviceState** out) {
    if (dev < 0 || dev >= kMaxDevices) return SEG_ERR_CUDA;
    DeviceState& ds = g_dev[dev];
    if (!ds.init) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SEG_ERR_CUDA;
        unsigned int* st = nullptr;
        if (cudaMalloc(&st, sizeof(unsigned int)) != cudaSuccess) {
            cudaGetLastError();
            return SEG_ERR_OUT_OF_MEMORY;
        }
        if (cudaMemset(st, 0, sizeof(unsigned int)) != cudaSuccess) return SEG_ERR_CUDA;
        ds.sm_count = sms;
        ds.status = st;
        ds.init = true;
    }
    *out = &ds;
    return SEG_OK;
}

// Scratch for (device, stream): grown on demand, zeroed when (re)allocated,
// stream-ordered so earlier work on the stream still sees the old buffer.
seg_status_t scratch_in(std::map<std::pair<int, cudaStream_t>, Scratch>& cache, int dev,
                        cudaStream_t stream, size_t bytes, Scratch** out) {
    Scratch& sc = cache[std::make_pair(dev, stream)];
    if (sc.bytes < bytes || sc.gen == UINT32_MAX) {
        size_t want = std::max<size_t>(bytes, size_t(1) << 20);
        want = std::max(want, sc.bytes);
        if (sc.ptr) cudaFreeAsync(sc.ptr, stream);
        sc.ptr = nullptr;
        sc.bytes = 0;
        if (cudaMallocAsync(&sc.ptr, want, stream) != cudaSuccess) {
            cudaGetLastError();
            sc.ptr = nullptr;
            return SEG_ERR_OUT_OF_MEMORY;
        }
        if (cudaMemsetAsync(sc.ptr, 0, want, stream) != cudaSuccess) return SEG_ERR_CUDA;
        sc.bytes = want;
        sc.gen = 0;
    }
    *out = &sc;
    return SEG_OK;
}

seg_status_t scratch_for(int dev, cudaStream_t stream, size_t bytes, Scratch** out) {
    return scratch_in(g_scratch, dev, stream, bytes, out);
}

// ---------------------------------------------------------------------------
// Fixed scratch for seg_reduce_noalloc: static device memory, one array per
// device (a __device__ variable exists once in every context), so that call
// never allocates.  Its ticket words must read zero before the first launch;
// set-up clears them once per device.

static __device__ __align__(256) unsigned char g_fixed_scratch[SEG_NOALLOC_SCRATCH_BYTES];
static __device__ unsigned int g_fixed_status;   // device errors when the caller passes no word

constexpr int kMaxKernels = 128;   // compiled kernels: 3 dtypes x 3 ops x 2 offset types x 7 shapes

struct FixedState {
    bool init = false;
    int sm_count = 0;
    unsigned char* scratch = nullptr;
    unsigned int* status = nullptr;
    uint32_t gen = 0;
    const void* configured[kMaxKernels] = {};
    int n_configured = 0;
};

std::mutex g_fixed_mu;
FixedState g_fixed[kMaxDevices];

// First call on a device: SM count, the arrays' addresses, zeroed ticket
// words (waited for, so that every later launch on any stream sees zeros).
seg_status_t fixed_state(int dev, cudaStream_t stream, FixedState** out) {
    if (dev < 0 || dev >= kMaxDevices) return SEG_ERR_CUDA;
    FixedState& fs = g_fixed[dev];
    if (!fs.init) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SEG_ERR_CUDA;
        void* scratch = nullptr;
        void* status = nullptr;
        if (cudaGetSymbolAddress(&scratch, g_fixed_scratch) != cudaSuccess ||
            cudaGetSymbolAddress(&status, g_fixed_status) != cudaSuccess) {
            cudaGetLastError();
            return SEG_ERR_CUDA;
        }
        const int64_t tickets = ticket_region_bytes(sms);
        if (tickets > int64_t(SEG_NOALLOC_SCRATCH_BYTES)) return SEG_ERR_SCRATCH_LIMIT;
        if (cudaMemsetAsync(scratch, 0, static_cast<size_t>(tickets), stream) != cudaSuccess ||
            cudaMemsetAsync(status, 0, sizeof(unsigned int), stream) != cudaSuccess ||
            cudaStreamSynchronize(stream) != cudaSuccess) {
            cudaGetLastError();
            return SEG_ERR_CUDA;
        }
        fs.sm_count = sms;
        fs.scratch = static_cast<unsigned char*>(scratch);
        fs.status = static_cast<unsigned int*>(status);
        fs.init = true;
    }
    *out = &fs;
    return SEG_OK;
}

// The offsets producers (run-length encoding, flags to offsets): the CTA
// count, scratch from the (device, stream) buffer past the ticket words
// (which these launches never touch), then the two launches.
seg_status_t run_producer(RleParams& p, int64_t n, int64_t* count, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SEG_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* ds = nullptr;
    seg_status_t st = device_state(dev, &ds);
    if (st != SEG_OK) return st;
    p.n = n;
    p.count = count;
    p.tiles = ceil_div(n, RLE_TILE);
    if (p.tiles > int64_t(INT32_MAX)) return SEG_ERR_UNSUPPORTED;   // tile indices stay 32-bit
    p.ctas = static_cast<int32_t>(std::min<int64_t>(
        p.tiles, std::min<int64_t>(int64_t(ds->sm_count) * RLE_CTAS_PER_SM, RLE_MAX_CTAS)));
    // scratch past the reduction's ticket words (which these launches never
    // touch): the per-CTA arrays, then the bitmap
    const int64_t ticket_bytes = ticket_region_bytes(ds->sm_count);
    Scratch* sc = nullptr;
    st = scratch_for(dev, stream,
                     static_cast<size_t>(ticket_bytes + RLE_CTA_SCRATCH + rle_tile_bytes(p.tiles)), &sc);
    if (st != SEG_OK) return st;
    int64_t* ws = reinterpret_cast<int64_t*>(static_cast<unsigned char*>(sc->ptr) + ticket_bytes);
    p.cta_count = ws;
    p.cta_first = ws + RLE_MAX_CTAS;
    p.tile_first = ws + 2 * RLE_MAX_CTAS;
    p.tile_count = reinterpret_cast<int32_t*>(p.tile_first + p.tiles);
    p.bitmap = reinterpret_cast<unsigned long long*>(
        reinterpret_cast<unsigned char*>(p.tile_first) + ((p.tiles * 12 + 255) / 256) * 256);
    static const char kProducerKey = 0;
    if (!ds->configured[&kProducerKey]) {
        if (configure_rle() != cudaSuccess) {
            cudaGetLastError();
            return SEG_ERR_CUDA;
        }
        ds->configured[&kProducerKey] = true;
    }
    if (launch_rle(p, stream) != cudaSuccess) {
        cudaGetLastError();
        return SEG_ERR_CUDA;
    }
    return SEG_OK;
}

}  // namespace

extern "C" {

seg_status_t seg_reduce_plan(seg_dtype_t dtype, int64_t F, int64_t num_values,
                             seg_offset_dtype_t offsets_dtype, int64_t num_segments, seg_op_t op,
                             uint64_t values_addr, int32_t sm_count, seg_plan_t* plan) {
    return plan_launch(dtype, F, num_values, offsets_dtype, num_segments, op, values_addr,
                       sm_count, plan);
}

seg_status_t seg_reduce(const void* values, seg_dtype_t dtype, int64_t F, int64_t num_values,
                        const void* offsets, seg_offset_dtype_t offsets_dtype,
                        int64_t num_segments, seg_op_t op, void* out, int64_t* out_arg,
                        seg_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const int64_t S = num_segments;
    // Host-visible argument checks; nothing is launched when one fails.
    if (dtype != SEG_U32 && dtype != SEG_S32 && dtype != SEG_F32) return SEG_ERR_INVALID_ARGUMENT;
    if (offsets_dtype != SEG_OFF_U32 && offsets_dtype != SEG_OFF_I64) return SEG_ERR_INVALID_ARGUMENT;
    if (op != SEG_SUM && op != SEG_MIN && op != SEG_MAX && op != SEG_MEAN) return SEG_ERR_INVALID_ARGUMENT;
    if (F < 1 || num_values < 0 || S < 0) return SEG_ERR_INVALID_ARGUMENT;
    if (op == SEG_MEAN && dtype != SEG_F32) return SEG_ERR_UNSUPPORTED;
    if (F > SEG_MAX_FEATURES) return SEG_ERR_UNSUPPORTED;
    if ((op == SEG_SUM || op == SEG_MEAN) && out_arg != nullptr) return SEG_ERR_INVALID_ARGUMENT;
    if (S == 0) return SEG_OK;
    if (!offsets || !out || (num_values > 0 && !values)) return SEG_ERR_INVALID_ARGUMENT;
    const size_t osz = offsets_dtype == SEG_OFF_U32 ? 4 : 8;
    if (reinterpret_cast<uintptr_t>(values) % 4 || reinterpret_cast<uintptr_t>(out) % 4 ||
        reinterpret_cast<uintptr_t>(offsets) % osz || reinterpret_cast<uintptr_t>(out_arg) % 8)
        return SEG_ERR_INVALID_ARGUMENT;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SEG_ERR_CUDA;

    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* ds = nullptr;
    seg_status_t st = device_state(dev, &ds);
    if (st != SEG_OK) return st;

    seg_plan_t pl;
    st = plan_launch(dtype, F, num_values, offsets_dtype, S, op,
                     reinterpret_cast<uint64_t>(values), ds->sm_count, &pl);
    if (st != SEG_OK) return st;

    const int kop = op == SEG_MIN ? OP_MIN : (op == SEG_MAX ? OP_MAX : OP_SUM);
    const int i64 = offsets_dtype == SEG_OFF_I64 ? 1 : 0;
    const void* fn = dtype == SEG_U32   ? pick_kernel_u32(kop, i64, pl.kernel_variant)
                     : dtype == SEG_S32 ? pick_kernel_s32(kop, i64, pl.kernel_variant)
                                        : pick_kernel_f32(kop, i64, pl.kernel_variant);
    if (!fn) return SEG_ERR_UNSUPPORTED;
    if (!ds->configured[fn]) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(pl.smem_bytes)) != cudaSuccess) {
            cudaGetLastError();
            return SEG_ERR_CUDA;
        }
        ds->configured[fn] = true;
    }

    Scratch* sc = nullptr;
    st = scratch_for(dev, stream, static_cast<size_t>(pl.workspace_bytes), &sc);
    if (st != SEG_OK) return st;
    sc->gen += 1;

    Params prm;
    prm.values = values;
    prm.offsets = offsets;
    prm.out = out;
    prm.out_arg = (op == SEG_MIN || op == SEG_MAX) ? out_arg : nullptr;
    prm.N = num_values;
    prm.S = S;
    prm.F = static_cast<int32_t>(F);
    prm.G = F > 1 ? pl.vecs_per_thread : 1;   // rows kernel: column slices
    prm.K = pl.items_per_slot;
    prm.max_ends = pl.max_ends;
    prm.P = pl.grid;
    prm.mean = op == SEG_MEAN ? 1 : 0;
    const int64_t ticket_bytes = ticket_region_bytes(ds->sm_count);
    prm.ws_tickets = static_cast<unsigned long long*>(sc->ptr);
    prm.ws_parts = static_cast<unsigned char*>(sc->ptr) + ticket_bytes;
    prm.status = ds->status;
    prm.gen = sc->gen;

    void* args[] = {&prm};
    const cudaError_t e = cudaLaunchKernel(fn, dim3(pl.grid), dim3(pl.block), args,
                                           static_cast<size_t>(pl.smem_bytes), stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SEG_ERR_CUDA;
    }
    return SEG_OK;
}

const char* seg_reduce_strerror(seg_status_t status) {
    switch (status) {
        case SEG_OK: return "success";
        case SEG_ERR_INVALID_ARGUMENT: return "invalid argument";
        case SEG_ERR_UNSUPPORTED: return "unsupported combination of arguments";
        case SEG_ERR_OUT_OF_MEMORY: return "out of device memory for scratch";
        case SEG_ERR_CUDA: return "CUDA runtime error";
        case SEG_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel ran out";
        case SEG_ERR_SCRATCH_LIMIT: return "the call needs more scratch than the fixed no-allocation array holds";
        default: return "unknown status";
    }
}

seg_status_t seg_reduce_device_status(seg_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (cudaStreamSynchronize(stream) != cudaSuccess) return SEG_ERR_CUDA;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SEG_ERR_CUDA;
    unsigned int* word = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        DeviceState* ds = nullptr;
        seg_status_t st = device_state(dev, &ds);
        if (st != SEG_OK) return st;
        word = ds->status;
    }
    unsigned int h = 0;
    if (cudaMemcpy(&h, word, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return SEG_ERR_CUDA;
    if (h != 0 && cudaMemset(word, 0, sizeof(h)) != cudaSuccess) return SEG_ERR_CUDA;
    return h ? SEG_ERR_DEVICE_TIMEOUT : SEG_OK;
}

seg_status_t seg_reduce_noalloc(const void* values, seg_dtype_t dtype, int64_t F,
                                int64_t num_values, const void* offsets,
                                seg_offset_dtype_t offsets_dtype, int64_t num_segments, seg_op_t op,
                                void* out, int64_t* out_arg, unsigned int* status_word,
                                seg_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const int64_t S = num_segments;
    // The same host-visible checks as seg_reduce; nothing is launched when one fails.
    if (dtype != SEG_U32 && dtype != SEG_S32 && dtype != SEG_F32) return SEG_ERR_INVALID_ARGUMENT;
    if (offsets_dtype != SEG_OFF_U32 && offsets_dtype != SEG_OFF_I64) return SEG_ERR_INVALID_ARGUMENT;
    if (op != SEG_SUM && op != SEG_MIN && op != SEG_MAX && op != SEG_MEAN) return SEG_ERR_INVALID_ARGUMENT;
    if (F < 1 || num_values < 0 || S < 0) return SEG_ERR_INVALID_ARGUMENT;
    if (op == SEG_MEAN && dtype != SEG_F32) return SEG_ERR_UNSUPPORTED;
    if (F > SEG_MAX_FEATURES) return SEG_ERR_UNSUPPORTED;
    if ((op == SEG_SUM || op == SEG_MEAN) && out_arg != nullptr) return SEG_ERR_INVALID_ARGUMENT;
    if (S == 0) return SEG_OK;
    if (!offsets || !out || (num_values > 0 && !values)) return SEG_ERR_INVALID_ARGUMENT;
    const size_t osz = offsets_dtype == SEG_OFF_U32 ? 4 : 8;
    if (reinterpret_cast<uintptr_t>(values) % 4 || reinterpret_cast<uintptr_t>(out) % 4 ||
        reinterpret_cast<uintptr_t>(offsets) % osz || reinterpret_cast<uintptr_t>(out_arg) % 8 ||
        reinterpret_cast<uintptr_t>(status_word) % 4)
        return SEG_ERR_INVALID_ARGUMENT;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SEG_ERR_CUDA;

    std::lock_guard<std::mutex> lock(g_fixed_mu);
    FixedState* fs = nullptr;
    seg_status_t st = fixed_state(dev, stream, &fs);
    if (st != SEG_OK) return st;

    seg_plan_t pl;
    st = plan_launch(dtype, F, num_values, offsets_dtype, S, op,
                     reinterpret_cast<uint64_t>(values), fs->sm_count, &pl);
    if (st != SEG_OK) return st;
    if (pl.workspace_bytes > int64_t(SEG_NOALLOC_SCRATCH_BYTES)) return SEG_ERR_SCRATCH_LIMIT;

    const int kop = op == SEG_MIN ? OP_MIN : (op == SEG_MAX ? OP_MAX : OP_SUM);
    const int i64 = offsets_dtype == SEG_OFF_I64 ? 1 : 0;
    const void* fn = dtype == SEG_U32   ? pick_kernel_u32(kop, i64, pl.kernel_variant)
                     : dtype == SEG_S32 ? pick_kernel_s32(kop, i64, pl.kernel_variant)
                                        : pick_kernel_f32(kop, i64, pl.kernel_variant);
    if (!fn) return SEG_ERR_UNSUPPORTED;
    bool configured = false;
    for (int k = 0; k < fs->n_configured; ++k) configured = configured || fs->configured[k] == fn;
    if (!configured) {
        if (fs->n_configured >= kMaxKernels) return SEG_ERR_UNSUPPORTED;
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(pl.smem_bytes)) != cudaSuccess) {
            cudaGetLastError();
            return SEG_ERR_CUDA;
        }
        fs->configured[fs->n_configured++] = fn;
    }
    // A new generation tag per call retires the previous call's ticket
    // counts; when the tag would wrap, the ticket words are cleared instead.
    if (fs->gen == UINT32_MAX) {
        if (cudaMemsetAsync(fs->scratch, 0, static_cast<size_t>(ticket_region_bytes(fs->sm_count)),
                            stream) != cudaSuccess) {
            cudaGetLastError();
            return SEG_ERR_CUDA;
        }
        fs->gen = 0;
    }
    fs->gen += 1;

    Params prm;
    prm.values = values;
    prm.offsets = offsets;
    prm.out = out;
    prm.out_arg = (op == SEG_MIN || op == SEG_MAX) ? out_arg : nullptr;
    prm.N = num_values;
    prm.S = S;
    prm.F = static_cast<int32_t>(F);
    prm.G = F > 1 ? pl.vecs_per_thread : 1;   // rows kernel: column slices
    prm.K = pl.items_per_slot;
    prm.max_ends = pl.max_ends;
    prm.P = pl.grid;
    prm.mean = op == SEG_MEAN ? 1 : 0;
    prm.ws_tickets = reinterpret_cast<unsigned long long*>(fs->scratch);
    prm.ws_parts = fs->scratch + ticket_region_bytes(fs->sm_count);
    prm.status = status_word != nullptr ? status_word : fs->status;
    prm.gen = fs->gen;

    void* args[] = {&prm};
    const cudaError_t e = cudaLaunchKernel(fn, dim3(pl.grid), dim3(pl.block), args,
                                           static_cast<size_t>(pl.smem_bytes), stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SEG_ERR_CUDA;
    }
    return SEG_OK;
}

seg_status_t seg_rle(const uint32_t* keys, int64_t n, uint32_t* values, uint32_t* lengths,
                     int64_t* offsets, int64_t* count, seg_stream_t stream) {
    if (n < 0 || n > int64_t(UINT32_MAX) || !count || (n > 0 && !keys)) return SEG_ERR_INVALID_ARGUMENT;
    if (reinterpret_cast<uintptr_t>(keys) % 4 || reinterpret_cast<uintptr_t>(values) % 4 ||
        reinterpret_cast<uintptr_t>(lengths) % 4 || reinterpret_cast<uintptr_t>(offsets) % 8 ||
        reinterpret_cast<uintptr_t>(count) % 8)
        return SEG_ERR_INVALID_ARGUMENT;
    RleParams p{};
    p.keys = keys;
    p.values = values;
    p.lengths = lengths;
    p.offsets = offsets;
    p.vec = reinterpret_cast<uintptr_t>(keys) % 16 == 0 ? 1 : 0;
    return run_producer(p, n, count, reinterpret_cast<cudaStream_t>(stream));
}

seg_status_t seg_flags_to_offsets(const uint8_t* flags, int64_t n, int64_t* offsets,
                                  int64_t* count, seg_stream_t stream) {
    if (n < 0 || !count || !offsets || (n > 0 && !flags)) return SEG_ERR_INVALID_ARGUMENT;
    if (reinterpret_cast<uintptr_t>(offsets) % 8 || reinterpret_cast<uintptr_t>(count) % 8)
        return SEG_ERR_INVALID_ARGUMENT;
    RleParams p{};
    p.flags = flags;
    p.flags_mode = 1;
    p.offsets = offsets;
    p.vec = reinterpret_cast<uintptr_t>(flags) % 16 == 0 ? 1 : 0;
    return run_producer(p, n, count, reinterpret_cast<cudaStream_t>(stream));
}

seg_status_t seg_reduce_sequential(const float* values, int64_t F, int64_t num_values,
                                   const void* offsets, seg_offset_dtype_t offsets_dtype,
                                   int64_t num_segments, seg_op_t op, float* out,
                                   seg_stream_t stream) {
    if (offsets_dtype != SEG_OFF_U32 && offsets_dtype != SEG_OFF_I64) return SEG_ERR_INVALID_ARGUMENT;
    if (op != SEG_SUM && op != SEG_MEAN) return SEG_ERR_INVALID_ARGUMENT;
    if (F < 1 || num_values < 0 || num_segments < 0) return SEG_ERR_INVALID_ARGUMENT;
    if (F > SEG_MAX_FEATURES) return SEG_ERR_UNSUPPORTED;
    if (num_segments == 0) return SEG_OK;
    if (!offsets || !out || (num_values > 0 && !values)) return SEG_ERR_INVALID_ARGUMENT;
    const size_t osz = offsets_dtype == SEG_OFF_U32 ? 4 : 8;
    if (reinterpret_cast<uintptr_t>(values) % 4 || reinterpret_cast<uintptr_t>(out) % 4 ||
        reinterpret_cast<uintptr_t>(offsets) % osz)
        return SEG_ERR_INVALID_ARGUMENT;
    if (offsets_dtype == SEG_OFF_U32 && num_values > int64_t(UINT32_MAX)) return SEG_ERR_INVALID_ARGUMENT;
    if (ceil_div(num_segments * F, SEQ_NT) > int64_t(INT32_MAX)) return SEG_ERR_UNSUPPORTED;
    SeqParams p{};
    p.values = values;
    p.offsets = offsets;
    p.off64 = offsets_dtype == SEG_OFF_I64 ? 1 : 0;
    p.mean = op == SEG_MEAN ? 1 : 0;
    p.N = num_values;
    p.F = F;
    p.S = num_segments;
    p.out = out;
    if (launch_sequential(p, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return SEG_ERR_CUDA;
    }
    return SEG_OK;
}

seg_status_t seg_scatter(const void* src, seg_dtype_t dtype, int64_t F, int64_t num_rows,
                         const int64_t* index, int64_t dim_size, seg_op_t op, void* out,
                         int64_t* out_arg, seg_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (dtype != SEG_U32 && dtype != SEG_S32 && dtype != SEG_F32) return SEG_ERR_INVALID_ARGUMENT;
    if (op != SEG_SUM && op != SEG_MIN && op != SEG_MAX && op != SEG_MEAN) return SEG_ERR_INVALID_ARGUMENT;
    if (F < 1 || num_rows < 0 || dim_size < 0) return SEG_ERR_INVALID_ARGUMENT;
    if (op == SEG_MEAN && dtype != SEG_F32) return SEG_ERR_UNSUPPORTED;
    if (F > SEG_MAX_FEATURES) return SEG_ERR_UNSUPPORTED;
    if ((op == SEG_SUM || op == SEG_MEAN) && out_arg != nullptr) return SEG_ERR_INVALID_ARGUMENT;
    // rows are packed into 32 bits next to the value for max / min
    if (num_rows >= int64_t(UINT32_MAX)) return SEG_ERR_UNSUPPORTED;
    if (dim_size == 0) return SEG_OK;
    if (!out || (num_rows > 0 && (!src || !index))) return SEG_ERR_INVALID_ARGUMENT;
    if (reinterpret_cast<uintptr_t>(src) % 4 || reinterpret_cast<uintptr_t>(out) % 4 ||
        reinterpret_cast<uintptr_t>(index) % 8 || reinterpret_cast<uintptr_t>(out_arg) % 8)
        return SEG_ERR_INVALID_ARGUMENT;
    if (ceil_div(dim_size * F, 8) > int64_t(INT32_MAX)) return SEG_ERR_UNSUPPORTED;
    // one launch covers every element (no grid-stride loop): at most 2^30 CTAs
    if (ceil_div(num_rows * F, int64_t(SC_NT) * SC_ITEMS) > (int64_t(1) << 30)) return SEG_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SEG_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* ds = nullptr;
    seg_status_t st = device_state(dev, &ds);
    if (st != SEG_OK) return st;
    ScatterParams p{};
    p.src = src;
    p.index = index;
    p.N = num_rows;
    p.F = F;
    p.D = dim_size;
    p.dtype = dtype == SEG_F32 ? 2 : (dtype == SEG_S32 ? 1 : 0);
    p.op = op == SEG_SUM ? 0 : (op == SEG_MIN ? 1 : (op == SEG_MAX ? 2 : 3));
    p.vec = (dtype == SEG_F32 && F % 4 == 0 && reinterpret_cast<uintptr_t>(src) % 16 == 0 &&
             reinterpret_cast<uintptr_t>(out) % 16 == 0) ? 4 : 1;
    p.out = out;
    p.arg = (op == SEG_MIN || op == SEG_MAX) ? out_arg : nullptr;
    const int64_t need = (op == SEG_MIN || op == SEG_MAX) ? dim_size * F * 8 : (op == SEG_MEAN ? dim_size * 4 : 0);
    if (need > 0) {
        // scratch past the reduction's ticket words, which these launches never touch
        const int64_t ticket_bytes = ticket_region_bytes(ds->sm_count);
        Scratch* sc = nullptr;
        st = scratch_for(dev, stream, static_cast<size_t>(ticket_bytes + need), &sc);
        if (st != SEG_OK) return st;
        unsigned char* ws = static_cast<unsigned char*>(sc->ptr) + ticket_bytes;
        if (op == SEG_MEAN) p.count = reinterpret_cast<uint32_t*>(ws);
        else p.word = reinterpret_cast<unsigned long long*>(ws);
    }
    if (launch_scatter(p, stream) != cudaSuccess) {
        cudaGetLastError();
        return SEG_ERR_CUDA;
    }
    return SEG_OK;
}

seg_status_t seg_scatter_sorted(const void* src, seg_dtype_t dtype, int64_t F, int64_t num_rows,
                                const int64_t* index, int64_t dim_size, seg_op_t op, void* out,
                                int64_t* out_arg, seg_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (dtype != SEG_U32 && dtype != SEG_S32 && dtype != SEG_F32) return SEG_ERR_INVALID_ARGUMENT;
    if (op != SEG_SUM && op != SEG_MIN && op != SEG_MAX && op != SEG_MEAN) return SEG_ERR_INVALID_ARGUMENT;
    if (F < 1 || num_rows < 0 || dim_size < 0) return SEG_ERR_INVALID_ARGUMENT;
    if (op == SEG_MEAN && dtype != SEG_F32) return SEG_ERR_UNSUPPORTED;
    if (F > SEG_MAX_FEATURES) return SEG_ERR_UNSUPPORTED;
    if ((op == SEG_SUM || op == SEG_MEAN) && out_arg != nullptr) return SEG_ERR_INVALID_ARGUMENT;
    // row numbers and keys are 32-bit
    if (num_rows >= int64_t(UINT32_MAX) || dim_size >= int64_t(UINT32_MAX)) return SEG_ERR_UNSUPPORTED;
    if (dim_size == 0) return SEG_OK;
    if (!out || (num_rows > 0 && (!src || !index))) return SEG_ERR_INVALID_ARGUMENT;
    if (reinterpret_cast<uintptr_t>(src) % 4 || reinterpret_cast<uintptr_t>(out) % 4 ||
        reinterpret_cast<uintptr_t>(index) % 8 || reinterpret_cast<uintptr_t>(out_arg) % 8)
        return SEG_ERR_INVALID_ARGUMENT;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SEG_ERR_CUDA;
    SortParams sp{};
    int64_t* offsets = nullptr;
    void* rows = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        DeviceState* ds = nullptr;
        seg_status_t st = device_state(dev, &ds);
        if (st != SEG_OK) return st;
        // sort buffers, then offsets, then the gathered rows
        const int64_t sort_bytes = ceil_div(sort_scratch_bytes(num_rows), 256) * 256;
        const int64_t off_bytes = ceil_div((dim_size + 1) * 8, 256) * 256;
        const int64_t row_bytes = num_rows * F * 4;
        Scratch* sc = nullptr;
        st = scratch_in(g_sort_scratch, dev, stream, static_cast<size_t>(sort_bytes + off_bytes + row_bytes), &sc);
        if (st != SEG_OK) return st;
        unsigned char* ws = static_cast<unsigned char*>(sc->ptr);
        sp.index = index;
        sp.N = num_rows;
        sp.D = dim_size;
        sp.tiles = ceil_div(num_rows, SORT_TILE);
        for (int b = 0; b < 2; ++b) {
            sp.keys[b] = reinterpret_cast<uint32_t*>(ws) + b * num_rows;
            sp.vals[b] = reinterpret_cast<uint32_t*>(ws) + (2 + b) * num_rows;
        }
        sp.hist = reinterpret_cast<uint32_t*>(ws) + 4 * num_rows;
        sp.total = sp.hist + int64_t(SORT_RADIX) * sp.tiles;
        int bits = 0;
        for (int64_t d = dim_size; d > 0; d >>= 1) ++bits;   // keys go up to dim_size
        sp.passes = (bits + 7) / 8;
        offsets = reinterpret_cast<int64_t*>(ws + sort_bytes);
        rows = ws + sort_bytes + off_bytes;
        const uint32_t* sorted = sp.keys[(sp.passes - 1) & 1];
        const uint32_t* perm = sp.vals[(sp.passes - 1) & 1];
        if (launch_sort(sp, stream) != cudaSuccess ||
            launch_bucket_offsets(sorted, num_rows, dim_size, offsets, stream) != cudaSuccess ||
            launch_gather_rows(src, perm, num_rows, F, rows, stream) != cudaSuccess) {
            cudaGetLastError();
            return SEG_ERR_CUDA;
        }
    }
    // the groups are contiguous now: the deterministic segmented reduction
    const seg_status_t st = seg_reduce(num_rows > 0 ? rows : nullptr, dtype, F, num_rows, offsets, SEG_OFF_I64,
                                       dim_size, op, out, out_arg, stream_);
    if (st != SEG_OK) return st;
    if (out_arg != nullptr && (op == SEG_MIN || op == SEG_MAX) && num_rows > 0) {
        // args name rows of the sorted copy: map them back to src's rows
        if (launch_map_args(out_arg, sp.vals[(sp.passes - 1) & 1], dim_size * F, stream) != cudaSuccess) {
            cudaGetLastError();
            return SEG_ERR_CUDA;
        }
    }
    return SEG_OK;
}

seg_status_t seg_scan(const void* values, seg_dtype_t dtype, int64_t num_values, const void* offsets,
                      seg_offset_dtype_t offsets_dtype, int64_t num_segments, seg_op_t op,
                      int32_t exclusive, void* out, seg_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (dtype != SEG_U32 && dtype != SEG_S32 && dtype != SEG_F32) return SEG_ERR_INVALID_ARGUMENT;
    if (offsets_dtype != SEG_OFF_U32 && offsets_dtype != SEG_OFF_I64) return SEG_ERR_INVALID_ARGUMENT;
    if (op != SEG_SUM && op != SEG_MIN && op != SEG_MAX) return SEG_ERR_INVALID_ARGUMENT;
    if (exclusive != 0 && exclusive != 1) return SEG_ERR_INVALID_ARGUMENT;
    if (exclusive && op != SEG_SUM) return SEG_ERR_UNSUPPORTED;
    if (num_values < 0 || num_segments < 0) return SEG_ERR_INVALID_ARGUMENT;
    if (num_values == 0) return SEG_OK;
    if (!values || !offsets || !out) return SEG_ERR_INVALID_ARGUMENT;
    const size_t osz = offsets_dtype == SEG_OFF_U32 ? 4 : 8;
    if (reinterpret_cast<uintptr_t>(values) % 4 || reinterpret_cast<uintptr_t>(out) % 4 ||
        reinterpret_cast<uintptr_t>(offsets) % osz)
        return SEG_ERR_INVALID_ARGUMENT;
    if (offsets_dtype == SEG_OFF_U32 && num_values > int64_t(UINT32_MAX)) return SEG_ERR_INVALID_ARGUMENT;
    const int64_t tiles = ceil_div(num_values, RS_TILE);
    if (tiles > int64_t(INT32_MAX)) return SEG_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SEG_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* ds = nullptr;
    seg_status_t st = device_state(dev, &ds);
    if (st != SEG_OK) return st;
    // scratch past the reduction's ticket words: per-CTA words, then the bitmap;
    // the ticket is slot 0 of the ticket words, tagged with a new generation
    const int64_t ticket_bytes = ticket_region_bytes(ds->sm_count);
    const int64_t cta_bytes = int64_t(RS_MAX_CTAS) * (8 + 8 + 8 + 4 + 4 + 4);
    const int64_t bitmap_bytes = rs_bitmap_words(num_values) * 8;
    Scratch* sc = nullptr;
    st = scratch_for(dev, stream, static_cast<size_t>(ticket_bytes + cta_bytes + bitmap_bytes), &sc);
    if (st != SEG_OK) return st;
    sc->gen += 1;
    unsigned char* ws = static_cast<unsigned char*>(sc->ptr) + ticket_bytes;
    ScanParams p{};
    p.values = values;
    p.offsets = offsets;
    p.off64 = offsets_dtype == SEG_OFF_I64 ? 1 : 0;
    p.dtype = dtype == SEG_F32 ? 2 : (dtype == SEG_S32 ? 1 : 0);
    p.op = op == SEG_SUM ? 0 : (op == SEG_MIN ? 1 : 2);
    p.exclusive = exclusive;
    p.vec = reinterpret_cast<uintptr_t>(values) % 16 == 0 && reinterpret_cast<uintptr_t>(out) % 16 == 0 ? 1 : 0;
    p.N = num_values;
    p.S = num_segments;
    p.out = out;
    p.tiles = tiles;
    p.sm_count = ds->sm_count;
    p.gen = sc->gen;
    p.ticket = static_cast<unsigned long long*>(sc->ptr);
    p.cta_aggf = reinterpret_cast<PartPair*>(ws);
    p.carryf = p.cta_aggf + RS_MAX_CTAS;
    p.cta_first = reinterpret_cast<int64_t*>(p.carryf + RS_MAX_CTAS);
    p.cta_aggi = reinterpret_cast<uint32_t*>(p.cta_first + RS_MAX_CTAS);
    p.carryi = p.cta_aggi + RS_MAX_CTAS;
    p.cta_flag = reinterpret_cast<int32_t*>(p.carryi + RS_MAX_CTAS);
    p.bitmap = reinterpret_cast<unsigned long long*>(ws + cta_bytes);
    if (launch_scan(p, stream) != cudaSuccess) {
        cudaGetLastError();
        return SEG_ERR_CUDA;
    }
    return SEG_OK;
}

seg_status_t seg_selftest_wait_timeout(uint32_t limit_ms, seg_stream_t stream_) {
    if (limit_ms < 1 || limit_ms > 10000) return SEG_ERR_INVALID_ARGUMENT;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SEG_ERR_CUDA;
    unsigned int* status = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        DeviceState* ds = nullptr;
        const seg_status_t st = device_state(dev, &ds);
        if (st != SEG_OK) return st;
        status = ds->status;
    }
    selftest_wait_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream_)>>>(
        status, static_cast<uint64_t>(limit_ms) * 1000000ull);
    if (cudaGetLastError() != cudaSuccess) return SEG_ERR_CUDA;
    return SEG_OK;
}

int32_t seg_reduce_version(void) { return kVersion; }

}  // extern "C"
