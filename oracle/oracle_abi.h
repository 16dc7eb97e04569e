/*
 * TEST INFRASTRUCTURE ONLY.  The CPU oracle of the gate-level re-simulator.
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may load it.
 * It shares no code with the CUDA library.
 *
 * Netlist arrays (all host memory, read only; same meaning as the arrays the
 * synthetic generator emits):
 *   nets 0..P-1 are primary/pseudo-primary inputs, gate g drives net P+g;
 *   gates are numbered in level order, level l holds [level_offsets[l], level_offsets[l+1]);
 *   gate g has pins fanin_off[g] .. fanin_off[g+1]-1 (in pin order);
 *   truth table of type t: tt_data[type_tt_off[t] .. + 2^n), indexed by the sum of
 *     pin_weight over the pins at 1 (GATSPI page, Fig. 4);
 *   delay table of gate g: dly_data[gate_dly_off[g] ...] laid out [4n][2^(n-1)],
 *     row 4*pin + 2*e_in + e_out (RISE = 0, FALL = 1), INT32_MAX = no arc.
 */
#ifndef GATSPI_ORACLE_ABI_H
#define GATSPI_ORACLE_ABI_H
#include <stdint.h>

typedef struct {
    int32_t num_inputs;
    int32_t num_gates;
    int32_t num_levels;
    int32_t num_types;
    const int32_t *level_offsets;
    const int32_t *gate_type;
    const int32_t *type_num_pins;
    const int32_t *type_tt_off;
    const uint8_t *tt_data;
    const int32_t *fanin_off;
    const int32_t *fanin_net;
    const int32_t *pin_weight;
    const int32_t *wire_rise;
    const int32_t *wire_fall;
    const int64_t *gate_dly_off;
    const int32_t *dly_data;
} oracle_netlist;

enum { ORACLE_OK = 0, ORACLE_EINVAL = 1, ORACLE_ENOMEM = 2, ORACLE_EBADWAVE = 4, ORACLE_EBADLUT = 7 };

#endif
