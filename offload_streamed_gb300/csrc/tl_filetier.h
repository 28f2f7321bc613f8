// tl_filetier.h -- the file tier of a streamed operator's weight store (host
// side).
//
// ZeRO-Infinity keeps what does not fit in host memory on NVMe and moves it
// up one tier at a time: NVMe -> pinned CPU buffers with direct I/O, then
// CPU -> GPU, each stage working on a different tile at the same time
// (ZeRO-Infinity, "Overlap-centric design"; memory-centric tiling,
// "Pitfalls").  Here W and dW live in files, tile-major [N][K][Mi] bf16.
// Reader threads fill a ring of pinned host slots from the W file with
// direct I/O, ahead of the engine's host->device copies; the engine's
// device->host copies of dW land in other pinned slots, which writer threads
// store to the dW file.  The engine asks for the tiles of each call in the
// order it will take them, so reads run ahead of the copies by up to the
// number of host slots, as the copies run ahead of the GEMMs by d.
#pragma once
#include <cstddef>
#include <cstdint>
#include <string>
#include <cuda_runtime.h>

namespace tl {

struct FileTierStats {
    int64_t read_bytes = 0, write_bytes = 0;
    double read_s = 0, write_s = 0;           // summed wall time of the tile reads / writes
    double fetch_wait_s = 0;                 // time the engine waited for a tile to be read
    double writeback_wait_s = 0;             // time the engine waited for a free dW slot
};

class FileTier {
public:
    // Opens w_path for reading (it must hold n_tiles * tile_bytes) and dw_path
    // for writing (created, and extended to that size), both with direct
    // I/O; tile_bytes must be a multiple of 4096.  Allocates host_slots (>= 2)
    // pinned slots for each direction and starts io_threads (>= 1) threads per
    // direction.  Needs the device current.  nullptr (and *why) on failure.
    static FileTier* open(const char* w_path, const char* dw_path, int32_t n_tiles, size_t tile_bytes,
                          int32_t host_slots, int32_t io_threads, std::string* why);
    ~FileTier();  // waits for the pending writes, then stops the threads and frees everything

    // Append tiles to the read order.
    void request(int32_t tile);
    // Block until the next tile of the read order is in a host slot; it must
    // be `tile`.  Returns the slot, or -1 on an I/O error or an order mismatch.
    int acquire_w(int32_t tile, std::string* why);
    const void* w_slot(int s) const;
    // Record this event after the copy that reads slot s, then release_w(s):
    // the slot is read into again once the event has completed.
    cudaEvent_t w_event(int s) const;
    void release_w(int s);
    // Drop the read order (after a failed call).
    void clear_requests();

    // Block until a dW slot is free (its last contents are in the file).
    int acquire_dw(std::string* why);
    void* dw_slot(int s) const;
    // Record this event after the copy that fills slot s, then commit_dw: a
    // writer stores the slot as tile `tile` once the event has completed.
    cudaEvent_t dw_event(int s) const;
    void commit_dw(int s, int32_t tile);
    // Block until every committed dW tile is in the file.
    bool sync(std::string* why);

    FileTierStats stats() const;
    int32_t host_slots() const;
    int32_t io_threads() const;

    struct Impl;

private:
    explicit FileTier(Impl* p) : p_(p) {}
    Impl* p_;
};

}  // namespace tl
