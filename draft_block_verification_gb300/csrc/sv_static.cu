// sv_static.cu -- greedy verification that allocates no device memory.
//
// sv_verify_greedy keeps its scratch (per-unit records, completion counters,
// control words) in a handle whose workspace grows with cudaMallocAsync.  Some
// callers cannot let a library allocate: a serving engine that reserves all
// free device memory for its own pools up front (a KV cache, say), or a
// memory-capped process in which an allocation mid-step could fail or force a
// synchronising defragmentation.  sv_verify_greedy_static runs the same
// streaming kernel with its scratch in one fixed, file-scope device array
// instead, and needs no handle.
//
// Limits (checked on the host; larger shapes are rejected with
// SV_ERR_UNSUPPORTED before anything is enqueued):
//   B <= kStaticMaxSeqs sequences and B * (K + 1) <= kStaticMaxRows rows.
// The scratch is about 2.1 MB per device.
//
// Calls on one device share that scratch, so they must not overlap: issue
// them on one stream, or order streams with events.  The first call on a
// device looks up the scratch address (cudaGetSymbolAddress) and sets the
// kernel attributes; make that first call before any stream capture.  A
// set-up that fails with a CUDA error is not remembered: the next call on
// that device tries again.
#include <cuda_runtime.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "sv_gumbel.cuh"
#include "sv_job.cuh"

namespace sv {
sv_status fault_injected(const char *call);
size_t pass_smem_bytes();
cudaError_t pass_setup(int *blocks_per_sm);
cudaError_t pass_launch(const Job &j, int grid, cudaStream_t s);
}  // namespace sv

using namespace sv;

namespace {

constexpr int kStaticMaxSeqs = 4096;
constexpr int kStaticMaxRows = 32768;
constexpr int kStaticMaxDevices = 64;

// Layout of the scratch: records, then control words and completion
// counters (zeroed by every call), then an all-zero bound table (the greedy
// rows never read it; the kernel only copies it to shared memory).
constexpr size_t kRecBytes = (size_t)kStaticMaxRows * sizeof(RowPart);
constexpr size_t kCntOff = kRecBytes;
constexpr size_t kCntWords = (size_t)C_NCTL + kStaticMaxSeqs;
constexpr size_t kTabOff = (kCntOff + kCntWords * sizeof(unsigned) + 255) & ~(size_t)255;
constexpr size_t kScratchBytes = kTabOff + kGTab * sizeof(float);

static __device__ __align__(256) unsigned char g_static_scratch[kScratchBytes];

struct DeviceSetup {
    bool done = false;            // set up successfully, or found unsupported
    sv_status status = SV_OK;     // SV_OK or SV_ERR_UNSUPPORTED once done
    unsigned char *scratch = nullptr;
    int sms = 0;
    int blocks_per_sm = 1;
};

std::mutex g_setup_mu;
DeviceSetup g_setup[kStaticMaxDevices];

// Once per device, with that device current.  Only a completed set-up and
// the finding that the device is not an sm_103 part are remembered: a CUDA
// error (for example a first call made inside a stream capture) is returned
// as SV_ERR_CUDA and the next call tries again.
sv_status setup_device(int dev, DeviceSetup **out)
{
    std::lock_guard<std::mutex> lk(g_setup_mu);
    DeviceSetup &d = g_setup[dev];
    *out = &d;
    if (d.done)
        return d.status;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
        return SV_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) {  // built for sm_103a only
        d.status = SV_ERR_UNSUPPORTED;
        d.done = true;
        return d.status;
    }
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    int nb = 0;
    if (e == cudaSuccess)
        e = pass_setup(&nb);
    if (e != cudaSuccess || p == nullptr)
        return SV_ERR_CUDA;
    d.sms = prop.multiProcessorCount;
    d.scratch = (unsigned char *)p;
    d.blocks_per_sm = std::max(nb, 1);
    d.status = SV_OK;
    d.done = true;
    return SV_OK;
}

bool logits_ok_static(const void *p, sv_dtype dt, int64_t rs, int V)
{
    if (!p || ((uintptr_t)p & 15u) != 0) return false;
    if (dt != SV_F32 && dt != SV_BF16) return false;
    const int esz = dt == SV_BF16 ? 2 : 4;
    if (V < 1 || (int64_t)V * esz % 16 != 0) return false;
    if (rs < V || (rs * esz) % 16 != 0) return false;
    return (int64_t)V <= (int64_t)1 << 30;
}

}  // namespace

extern "C" sv_status sv_verify_greedy_static(const void *target, sv_dtype dtype,
                                             int64_t row_stride, int B, int K, int V,
                                             const int32_t *draft_ids, const int32_t *draft_len,
                                             int32_t *accept_len, int32_t *next_token,
                                             int32_t *status, void *stream)
{
    if (B < 0 || K < 0 || K > kMaxK || !status) return SV_ERR_INVALID_ARG;
    if (B == 0)  // nothing to verify; the status word still reads 0
        return cudaMemsetAsync(status, 0, sizeof(int32_t), (cudaStream_t)stream) == cudaSuccess
                   ? SV_OK
                   : SV_ERR_CUDA;
    if (!logits_ok_static(target, dtype, row_stride, V) || !accept_len || !next_token ||
        (K > 0 && !draft_ids))
        return SV_ERR_INVALID_ARG;
    const long long rows = (long long)B * (K + 1);
    if (B > kStaticMaxSeqs || rows > kStaticMaxRows) return SV_ERR_UNSUPPORTED;
    if (sv_status fi = fault_injected("sv_verify_greedy_static")) return fi;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kStaticMaxDevices)
        return SV_ERR_UNSUPPORTED;
    DeviceSetup *d = nullptr;
    const sv_status st = setup_device(dev, &d);
    if (st != SV_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    unsigned *cnt = (unsigned *)(d->scratch + kCntOff);
    // The control words and counters start every call at zero; so does the
    // caller's status word, which then holds the first device-side error.
    cudaError_t e = cudaMemsetAsync(cnt, 0, ((size_t)C_NCTL + B) * sizeof(unsigned), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) return SV_ERR_CUDA;

    Job j;
    memset(&j, 0, sizeof j);
    const int esz = dtype == SV_BF16 ? 2 : 4;
    j.kind = K_GREEDY;
    j.dtype = dtype;
    j.src0 = (const char *)target;
    j.rs = row_stride * esz;
    j.V = V;
    j.nvec = (int)((int64_t)V * esz / 16);
    j.B = B;
    j.K = K;
    j.c1 = 1.4426950408889634f;
    j.eos = -1;
    j.ids = draft_ids;
    j.lens = draft_len;
    j.acc = accept_len;
    j.next = next_token;
    j.err = status;
    j.ctl = cnt;
    j.seq_done = cnt + C_NCTL;
    j.gtab = (const float *)(d->scratch + kTabOff);
    j.rp = (RowPart *)d->scratch;
    // Row split as in the handle path, capped by the record capacity.
    const int resident = d->sms * d->blocks_per_sm;
    const int max_parts = std::max(1, (j.nvec + kStageVecs - 1) / kStageVecs);
    long long want = (4LL * resident + rows - 1) / rows;
    want = std::min<long long>(want, kStaticMaxRows / rows);
    const int parts = (int)std::min<long long>(std::max<long long>(want, 1),
                                               std::min(max_parts, 16));
    j.rows_per_seq = K + 1;
    j.part_vecs = (j.nvec + parts - 1) / parts;
    j.parts = (j.nvec + j.part_vecs - 1) / j.part_vecs;
    j.total_units = rows * j.parts;
    e = pass_launch(j, resident, s);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
