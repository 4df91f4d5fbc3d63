"""Occupancy, written out plainly from the KernelScope backend doc,
occupancy/calculator.py — calculate_occupancy and GPU_SPECS.

TEST INFRASTRUCTURE ONLY (like the rest of oracle/): the reference the
library's ks_occupancy is compared with. Shares no code with the library.
"""

# (max threads, max warps, max blocks, registers, shared memory) per SM.
# The page prints sm_75 and sm_80 in full and elides the registers and shared
# memory of sm_86 / sm_89 and the registers of sm_90 ("..."): those, and the
# two Blackwell entries that are not on the page, are the public CUDA values.
SPECS = {
    "sm_75": (1024, 32, 16, 65536, 65536),
    "sm_80": (2048, 64, 32, 65536, 167936),
    "sm_86": (1536, 48, 16, 65536, 102400),
    "sm_89": (1536, 48, 24, 65536, 102400),
    "sm_90": (2048, 64, 32, 65536, 232448),
    "sm_100": (2048, 64, 32, 65536, 233472),
    "sm_103": (2048, 64, 32, 65536, 233472),
}


def occupancy(arch, threads_per_block, registers_per_thread, shared_memory_per_block=0):
    max_threads, max_warps, max_blocks, regs_per_sm, smem_per_sm = SPECS[arch]
    warps_per_block = (threads_per_block + 31) // 32
    # 1. registers, allocated per warp in groups of 256
    if registers_per_thread > 0:
        regs_per_warp = registers_per_thread * 32
        regs_per_warp = ((regs_per_warp + 255) // 256) * 256
        warps_by_regs = regs_per_sm // regs_per_warp
    else:
        warps_by_regs = max_warps
    # 2. shared memory, allocated per block in 256-byte chunks
    if shared_memory_per_block > 0:
        smem_per_block = ((shared_memory_per_block + 255) // 256) * 256
        blocks_by_smem = smem_per_sm // smem_per_block
        warps_by_smem = blocks_by_smem * warps_per_block
    else:
        warps_by_smem = max_warps
    # 3. block size
    blocks_by_threads = max_threads // threads_per_block
    max_blocks_now = min(blocks_by_threads, max_blocks)
    warps_by_block_size = max_blocks_now * warps_per_block
    active = min(warps_by_regs, warps_by_smem, warps_by_block_size)
    active = min(active, max_warps)
    if active == warps_by_regs:
        limiter = "registers"
    elif active == warps_by_smem:
        limiter = "shared_memory"
    else:
        limiter = "block_size"
    return {"active_warps_per_sm": active, "max_warps_per_sm": max_warps,
            "occupancy_percent": active / max_warps * 100, "limiter": limiter,
            "warps_by_registers": warps_by_regs, "warps_by_shared_memory": warps_by_smem,
            "warps_by_block_size": warps_by_block_size}
