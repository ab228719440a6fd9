// Test helper: prints the shared-memory plan of every forward-kernel instance
// (compile-time constants of the kernel's Cfg) from host code; needs no GPU.
#include <cstdio>

#include "fa_fwd_kernel.cuh"

template <int D, bool FP8, bool PAIR>
void show(const char* name) {
    using C = fa::Cfg<D, FP8, PAIR>;
    std::printf("%s tile_bytes=%d slot_bytes=%d stages=%d tiles=%d stage_bytes=%d smem_bytes=%d\n",
                name, C::kTileBytes, C::kSlotBytes, C::kStages, fa::kTiles, C::kStageBytes,
                C::kSmemBytes);
}

int main() {
    show<128, false, false>("bf16_d128");
    show<64, false, false>("bf16_d64");
    show<128, true, false>("e4m3_d128");
    show<128, false, true>("pair_bf16_d128");
    return 0;
}
