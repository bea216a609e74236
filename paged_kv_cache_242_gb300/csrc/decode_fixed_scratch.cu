// pkv_paged_decode_attention_fixed_scratch: the decode attention entry point
// for callers that cannot allocate device memory.
//
// Who needs it.  Some callers are handed device pointers by a host
// application that owns every allocation on the GPU (an inference server
// that gives its plugins only pre-registered buffers, or a runtime with its
// own memory pool and a fixed budget).  Such a caller may not call
// cudaMalloc itself: an unplanned allocation can fail under the host's
// budget, fragments the pool the host manages, and cudaMalloc / cudaFree can
// synchronise the device in the middle of the host's schedule.  The split
// (long-sequence) mode of pkv_paged_decode_attention needs a scratch buffer
// for per-partition statistics, so this entry point supplies it from a
// fixed array compiled into the library.
//
// The scratch is the file-scope device array below, PKV_FIXED_SCRATCH_BYTES
// (16 MiB) on every GPU that loads this library, held until the process
// exits.  Host code cannot use the array's name as a device address: the
// device address is looked up with cudaGetSymbolAddress, once per device,
// with that device current, on the first call that needs it (so make that
// first call on each device before any stream capture).  Every call shares
// the one array, so calls whose kernels overlap on the GPU (different
// streams, or different host threads) race on it; order them on one stream.
// Nothing in the array has to start at zero: the partition kernel writes
// every entry the merge kernel reads, in the same call.
#include <mutex>

#include "pkv_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_fixed_scratch[PKV_FIXED_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mutex;
void* g_scratch_address[kMaxDevices] = {};

// Device address of g_fixed_scratch on the current device (looked up once).
cudaError_t fixed_scratch_address(void** address) {
    int device = -1;
    cudaError_t err = cudaGetDevice(&device);
    if (err != cudaSuccess) return err;
    if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_address[device] == nullptr) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_fixed_scratch);
        if (err != cudaSuccess) return err;
        g_scratch_address[device] = p;
    }
    *address = g_scratch_address[device];
    return cudaSuccess;
}

}  // namespace

extern "C" pkv_status pkv_paged_decode_attention_fixed_scratch(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t max_seq_len, int32_t num_seqs,
    int32_t num_q_heads, pkv_cache_desc c, float scale, int32_t partition_size, void* out,
    int32_t* err_flag, void* stream) {
    const size_t need = pkv_decode_workspace_bytes(num_seqs, num_q_heads, c.head_dim, max_seq_len,
                                                   c.block_size, partition_size);
    if (need > PKV_FIXED_SCRATCH_BYTES) return PKV_ERR_WORKSPACE_TOO_SMALL;
    void* scratch = nullptr;
    if (need > 0 && fixed_scratch_address(&scratch) != cudaSuccess) return PKV_ERR_CUDA;
    return pkv_paged_decode_attention(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                      seq_lens, max_seq_len, num_seqs, num_q_heads, c, scale,
                                      partition_size, scratch,
                                      need > 0 ? PKV_FIXED_SCRATCH_BYTES : 0, out, err_flag,
                                      stream);
}
