// common.cuh -- geometry constants and host-side helpers shared by the library's
// translation units (error text, launch checks, TMA descriptor creation).
#pragma once
#include <cstdint>
#include <cstdio>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/k3mla.h"

namespace k3 {

constexpr int H = K3MLA_HEADS;          // 96
constexpr int NOPE = K3MLA_QK_NOPE;     // 128
constexpr int ROPE = K3MLA_QK_ROPE;     // 64
constexpr int QDIM = NOPE + ROPE;       // 192
constexpr int VH = K3MLA_V_HEAD;        // 128
constexpr int LORA = K3MLA_KV_LORA;     // 512
constexpr int ROW = K3MLA_ROW;          // 576
constexpr int PAGE = K3MLA_PAGE;        // 64
constexpr int TILE = K3MLA_TILE;        // 128
constexpr int WROWS_PER_HEAD = NOPE + VH;  // 256

// Per-thread error text for k3mla_last_error().
void set_error(const char* fmt, ...);

// Check a kernel launch; returns K3MLA_OK or K3MLA_E_CUDA with the text recorded.
int check_launch(const char* what);

// True if the current device is an sm_103 part; records the reason otherwise.
bool device_ok();

// 2-D bf16 tensor map over `rows` rows of `cols` elements (row pitch = cols*2
// bytes) with a box of box_cols x box_rows and 128-byte swizzle.
int make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                      uint32_t box_rows);

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace k3
