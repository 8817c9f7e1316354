"""MoE expert grouped GEMM on the NVFP4 library: weight preparation and the
decode/prefill call sequence.

Everything here is argument marshalling around the C ABI; the arithmetic
runs in the CUDA kernels.  Buffers are allocated once per plan (torch
device memory) so that a step enqueues kernels only.

Call sequence of one MoE pass ("The FP4 Frontier", Finding 5: grouped GEMM
over all experts; the activations arrive in BF16 and are quantised on the
fly, "The SM120 FP4 GEMM Kernel Investigation", The Context):
    route -> quantise + dispatch to route order -> grouped GEMM
    [-> weighted combine back to token order for the down projection]
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import nvfp4 as F


@dataclass
class ExpertWeights:
    """NVFP4 expert weights as operand tiles over [E*N, K], one global per expert."""
    tiles: torch.Tensor
    g: torch.Tensor
    E: int
    N: int
    K: int
    sparse: bool = False      # tiles are 2:4-sparse tiles (nvfp4_grouped_gemm_sparse)


def quantize_experts(w: torch.Tensor, stream=None) -> ExpertWeights:
    """BF16 [E, N, K] on the device -> NVFP4 operand tiles, one global per expert."""
    E, N, K = w.shape
    dev = w.device
    packed = torch.empty((E, N, K // 2), dtype=torch.uint8, device=dev)
    sf_rm = torch.empty((E, N, K // 16), dtype=torch.uint8, device=dev)
    g = torch.empty(E, dtype=torch.float32, device=dev)
    for e in range(E):
        F.nvfp4_quantize(w[e], packed[e], sf_rm[e], g[e:e + 1], 0, stream)
    tiles = torch.empty(F.nvfp4_operand_tiles_bytes(E * N, K), dtype=torch.uint8, device=dev)
    F.nvfp4_prepack_weight_tiles(packed.view(E * N, K // 2), sf_rm.view(E * N, K // 16), tiles,
                                 stream)
    return ExpertWeights(tiles, g, E, N, K)


@dataclass
class PlainExpertWeights:
    """NVFP4 expert weights in the plain layouts nvfp4_grouped_gemm takes:
    packed codes [E*N, K/2] and their scales in the tensor-core atom layout."""
    packed: torch.Tensor
    sf_atoms: torch.Tensor
    g: torch.Tensor
    E: int
    N: int
    K: int


def quantize_experts_plain(w: torch.Tensor, stream=None) -> PlainExpertWeights:
    """BF16 [E, N, K] on the device -> packed codes + atom-layout scales, one
    global per expert (nvfp4_quantize per expert, then nvfp4_prepack_weights
    over all E*N rows)."""
    E, N, K = w.shape
    dev = w.device
    packed = torch.empty((E * N, K // 2), dtype=torch.uint8, device=dev)
    sf_rm = torch.empty((E * N, K // 16), dtype=torch.uint8, device=dev)
    g = torch.empty(E, dtype=torch.float32, device=dev)
    for e in range(E):
        F.nvfp4_quantize(w[e], packed[e * N:(e + 1) * N], sf_rm[e * N:(e + 1) * N], g[e:e + 1],
                         0, stream)
    atoms = torch.empty(F.nvfp4_prepacked_scales_bytes(E * N, K // 16), dtype=torch.uint8,
                        device=dev)
    F.nvfp4_prepack_weights(sf_rm, atoms, stream)
    return PlainExpertWeights(packed, atoms, g, E, N, K)


def quantize_experts_sparse(w: torch.Tensor, stream=None, pruned: bool = False) -> ExpertWeights:
    """BF16 [E, N, K] on the device -> 2:4-sparse NVFP4 tiles ("The FP4
    Frontier", Finding 6): each expert pruned to 2:4 over element pairs (unless
    `pruned` says it already is), quantised with its own global, packed as
    sparse tiles (two thirds of the dense bytes)."""
    E, N, K = w.shape
    dev = w.device
    if not pruned:
        w = w.contiguous().clone()
        F.nvfp4_prune_2of4(w.view(E * N, K), w.view(E * N, K), stream)
    packed = torch.empty((E, N, K // 2), dtype=torch.uint8, device=dev)
    sf_rm = torch.empty((E, N, K // 16), dtype=torch.uint8, device=dev)
    g = torch.empty(E, dtype=torch.float32, device=dev)
    for e in range(E):
        F.nvfp4_quantize(w[e], packed[e], sf_rm[e], g[e:e + 1], 0, stream)
    tiles = torch.empty(F.nvfp4_sparse_tiles_bytes(E * N, K), dtype=torch.uint8, device=dev)
    F.nvfp4_prepack_sparse_weight_tiles(packed.view(E * N, K // 2), sf_rm.view(E * N, K // 16),
                                        tiles, stream)
    return ExpertWeights(tiles, g, E, N, K, sparse=True)


class GroupedPlan:
    """Buffers and calls for one grouped-GEMM shape.

    mode "gather": activations [T, K] in token order, each token quantised
    once and written to its top-k route positions; output [R, N] in route
    order.  mode "combine": activations [R, K] already in route order;
    output [T, N] = sum of the token's routes weighted by topk_weights.
    """

    def __init__(self, w: ExpertWeights, T: int, topk: int, mode: str, device="cuda",
                 routing_from: "GroupedPlan" = None, out: bool = True):
        assert mode in ("gather", "combine")
        self.w, self.T, self.topk, self.mode = w, T, topk, mode
        E, N, K = w.E, w.N, w.K
        R = T * topk
        self.R = R
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        if routing_from is not None:       # share one routing between two projections
            assert routing_from.T == T and routing_from.topk == topk and routing_from.w.E == E
            self.expert_offsets = routing_from.expert_offsets
            self.route_token = routing_from.route_token
            self.route_slot = routing_from.route_slot
            self.route_pos = routing_from.route_pos
        else:
            self.expert_offsets = torch.empty(E + 1, **i32)
            self.route_token = torch.empty(max(R, 1), **i32)
            self.route_slot = torch.empty(max(R, 1), **i32)
            self.route_pos = torch.empty(max(R, 1), **i32)
        self.a_tiles = torch.empty(max(F.nvfp4_grouped_tiles_bytes(R, E, K), 16),
                                   dtype=torch.uint8, device=dev)
        self.a_g = torch.empty(1, dtype=torch.float32, device=dev)
        if mode == "gather":
            # out=False: the plan only routes and quantises (its GEMM output
            # goes elsewhere, e.g. the fused MLP's h tiles)
            self.out = (torch.empty((max(R, 1), N), dtype=torch.bfloat16, device=dev)
                        if out else None)
            self.workspace = None
        else:
            self.out = torch.empty((max(T, 1), N), dtype=torch.bfloat16, device=dev)
            self.workspace = torch.empty(max(F.nvfp4_combine_workspace_bytes(T, N) // 4, 4),
                                         dtype=torch.float32, device=dev)

    def route(self, topk_ids, stream=None):
        F.nvfp4_moe_route(topk_ids, self.w.E, self.expert_offsets, self.route_token,
                          self.route_slot, self.route_pos, stream)

    def amax(self, x, stream=None):
        """The tensor amax half of quantize(); needs no routing."""
        F.nvfp4_amax_partials(x, self.R, self.w.E, self.a_tiles, stream)

    def quantize(self, x, stream=None, amax_done: bool = False):
        flags = F.NVFP4_AMAX_DONE if amax_done else 0
        if self.mode == "gather":
            F.nvfp4_quantize_dispatch(x, self.route_pos, self.topk, self.expert_offsets,
                                      self.w.E, self.R, self.a_tiles, self.a_g, flags, stream)
        else:
            F.nvfp4_quantize_dispatch(x, None, 1, self.expert_offsets, self.w.E, self.R,
                                      self.a_tiles, self.a_g, flags, stream)

    def gemm(self, topk_weights=None, stream=None):
        w = self.w
        fn = F.nvfp4_grouped_gemm_sparse if w.sparse else F.nvfp4_grouped_gemm_tiles
        fn(self.a_tiles, self.a_g, w.tiles, w.g,
                             self.expert_offsets, w.E, self.T, self.topk, w.N, w.K,
                             self.route_token, self.route_slot,
                             topk_weights if self.mode == "combine" else None,
                             self.out, self.workspace, stream)

    def run(self, x, topk_ids=None, topk_weights=None, stream=None, route=True):
        """route (optional) -> quantise/dispatch -> grouped GEMM (-> combine)."""
        if route:
            self.route(topk_ids, stream)
        self.quantize(x, stream)
        self.gemm(topk_weights, stream)
        return self.out


def _route_and_amax(plan: "GroupedPlan", x, topk_ids, side, stream=None):
    """Routing and the amax of x need nothing from each other: the amax runs
    on `side` while the routing runs on the step's stream, which then waits
    for it (fork and join by events, which CUDA graph capture records)."""
    main = torch.cuda.current_stream() if stream is None else stream
    side.wait_stream(main)
    with torch.cuda.stream(side):
        plan.amax(x, side)
    plan.route(topk_ids, main)
    main.wait_stream(side)


class DecodeLayer:
    """One MoE pass over a token batch: gate_up (gather) then down (combine).

    The down projection's input is a separate route-ordered BF16 tensor
    (the SiLU-and-multiply between the two projections is not part of this
    path), and both projections share one routing.
    """

    def __init__(self, w_gate_up: ExpertWeights, w_down: ExpertWeights, T: int, topk: int,
                 device="cuda"):
        self.gate_up = GroupedPlan(w_gate_up, T, topk, "gather", device)
        self.down = GroupedPlan(w_down, T, topk, "combine", device, routing_from=self.gate_up)
        self._side = torch.cuda.Stream(device=torch.device(device))
        self._side_h = torch.cuda.Stream(device=torch.device(device))

    def step(self, x, topk_ids, h, topk_weights, stream=None, timing=None):
        """x [T, K1] BF16, topk_ids [T, k] int32, h [R, K2] BF16 (route order),
        topk_weights [T, k] FP32 -> (gate_up out [R, N1], down out [T, N2]).

        h is an input of its own, so its quantisation (amax, then dispatch
        into the down projection's tiles) needs only the routing: it runs on
        a side stream beside x's quantisation and the gate_up GEMM, and the
        down GEMM waits for it (fork and join by events, which CUDA graph
        capture records).  `timing`, if given, is a pair of (start, end)
        CUDA-event lists that bracket the two grouped-GEMM calls."""
        gu, dn = self.gate_up, self.down
        main = torch.cuda.current_stream() if stream is None else stream
        _route_and_amax(gu, x, topk_ids, self._side, stream)
        self._side_h.wait_stream(main)              # after the routing
        with torch.cuda.stream(self._side_h):
            dn.quantize(h, self._side_h)
        gu.quantize(x, stream, amax_done=True)
        if timing is not None:
            timing[0][0].record()
        gu.gemm(None, stream)
        if timing is not None:
            timing[0][1].record()
        main.wait_stream(self._side_h)
        if timing is not None:
            timing[1][0].record()
        dn.gemm(topk_weights, stream)
        if timing is not None:
            timing[1][1].record()
        return gu.out, dn.out


class FusedMLP:
    """One expert MLP pass: route, quantise + dispatch x, then gate_up,
    SiLU(gate) * up and the NVFP4 quantisation of h in one grouped GEMM launch
    (nvfp4_moe_gate_up_silu), then the down projection with the weighted
    combine.  h never exists in BF16; its global scale g_h is given (a device
    float, calibrated by the caller).

    g_h=None selects the two-phase form: the gate_up launch writes h in BF16
    (nvfp4_moe_gate_up_silu_bf16), the dispatch quantiser finds its global from
    its amax and writes the down projection's tiles.

    single_launch=True (with a given g_h) runs gate_up, SiLU * up, the NVFP4
    quantisation of h, the down projection and the combine in one persistent
    launch (nvfp4_moe_mlp).
    """

    def __init__(self, w_gate_up: ExpertWeights, w_down: ExpertWeights, T: int, topk: int,
                 g_h: torch.Tensor = None, device="cuda", single_launch: bool = False):
        assert w_gate_up.E == w_down.E and w_gate_up.N == 2 * w_down.K
        assert not (single_launch and g_h is None), "one launch needs the global of h"
        self.w1, self.w2, self.T, self.topk, self.g_h = w_gate_up, w_down, T, topk, g_h
        self.single_launch = single_launch
        dev = torch.device(device)
        self.gate_up = GroupedPlan(w_gate_up, T, topk, "gather", device, out=False)
        self.down = GroupedPlan(w_down, T, topk, "combine", device, routing_from=self.gate_up)
        self.h = (torch.empty((max(T * topk, 1), w_down.K), dtype=torch.bfloat16, device=dev)
                  if g_h is None else None)
        self.mlp_ws = (torch.empty(max(F.nvfp4_moe_mlp_workspace_bytes(T, topk, w_down.E,
                                                                      w_down.N), 16),
                                   dtype=torch.uint8, device=dev) if single_launch else None)
        self._side = torch.cuda.Stream(device=dev)

    def step(self, x, topk_ids, topk_weights, stream=None):
        """x [T, K1] BF16, topk_ids [T, k] int32, topk_weights [T, k] FP32 ->
        out [T, N2] BF16 (the down plan's output buffer)."""
        gu, dn, w1, w2 = self.gate_up, self.down, self.w1, self.w2
        _route_and_amax(gu, x, topk_ids, self._side, stream)
        gu.quantize(x, stream, amax_done=True)
        if self.single_launch:
            F.nvfp4_moe_mlp(gu.a_tiles, gu.a_g, w1.tiles, w1.g, w2.tiles, w2.g, gu.expert_offsets,
                            w1.E, self.T, self.topk, w1.N, w1.K, w2.N, self.g_h, dn.a_tiles,
                            dn.route_token, dn.route_slot, topk_weights, dn.out, self.mlp_ws,
                            stream)
            return dn.out
        if self.g_h is not None:
            F.nvfp4_moe_gate_up_silu(gu.a_tiles, gu.a_g, w1.tiles, w1.g, gu.expert_offsets, w1.E,
                                     self.T, self.topk, w1.N, w1.K, self.g_h, dn.a_tiles, stream)
            g_h = self.g_h
        else:
            F.nvfp4_moe_gate_up_silu_bf16(gu.a_tiles, gu.a_g, w1.tiles, w1.g, gu.expert_offsets,
                                          w1.E, self.T, self.topk, w1.N, w1.K, self.h, stream)
            dn.quantize(self.h, stream)
            g_h = dn.a_g
        F.nvfp4_grouped_gemm_tiles(dn.a_tiles, g_h, w2.tiles, w2.g, dn.expert_offsets, w2.E,
                                   self.T, self.topk, w2.N, w2.K, dn.route_token, dn.route_slot,
                                   topk_weights, dn.out, dn.workspace, stream)
        return dn.out


class CapturedStep:
    """A DecodeLayer step recorded once into a CUDA graph over fixed input
    buffers; replay() re-runs every kernel of the step with one launch.

    The library's per-device set-up runs on the first eager call, so call
    the layer's step() at least once before capturing.
    """

    def __init__(self, layer: DecodeLayer, x, topk_ids, h, topk_weights):
        self.inputs = (x, topk_ids, h, topk_weights)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            layer.step(*self.inputs)
        torch.cuda.current_stream().wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.outputs = layer.step(*self.inputs)

    def replay(self):
        self.graph.replay()
        return self.outputs
