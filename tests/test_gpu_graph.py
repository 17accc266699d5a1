"""CUDA-graph capture of the decode path: a serving loop records its per-layer attention calls once
and replays them.  The calls issue only kernel launches on the given stream (the partition kernel
under programmatic dependent launch, then the merge), so a captured sequence of fused write +
decode calls must replay to the same bits as the same calls run eagerly."""
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def bits(t):
    return t.view(torch.int16)


@pytest.mark.parametrize("lens_kind", ["serving", "short"])
def test_captured_layer_loop_replays_to_the_eager_bits(cuda_lib, lens_kind):
    pa = cuda_lib
    dev = torch.device("cuda", 0)
    if lens_kind == "serving":
        lens = W.llama_context_lens()[:16]  # 16 sequences of 512-4096 tokens: split-K + merge
        num_blocks, max_blocks = 6000, W.LLAMA_MAX_CTX // 16
    else:
        lens = [1, 17, 200, 63, 900]       # short rows: single partitions and small splits
        num_blocks, max_blocks = 200, 64
    layers = 4
    inp = W.device_decode_inputs(lens, n_q_heads=32, n_kv_heads=8, head_dim=128, block_size=16,
                                 dtype=torch.bfloat16, num_blocks=num_blocks, max_blocks_per_seq=max_blocks,
                                 device=dev, seed=77, layers=layers)
    table, ctx, slot = inp["block_table"].to(dev), inp["context_lens"].to(dev), inp["slot_mapping"].to(dev)
    q, kn, vn = inp["q"].to(dev), inp["k_new"].to(dev), inp["v_new"].to(dev)
    B = len(lens)
    nbytes = pa.decode_workspace_size(B, table.stride(0), 16, 32, 8, 128)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev) if nbytes else None
    outs_eager = [torch.empty_like(q) for _ in range(layers)]
    outs_graph = [torch.empty_like(q) for _ in range(layers)]
    stream = torch.cuda.Stream()

    def run(outs):
        for layer in range(layers):
            kp, vp = inp["pools"][layer]
            pa.paged_attention_decode_fused(q, kn, vn, slot, kp, vp, table, ctx, out=outs[layer],
                                            workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        run(outs_eager)  # eager (also the warm-up: one-time attribute and tensor-map set-up)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        run(outs_graph)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    for layer in range(layers):
        assert torch.equal(bits(outs_graph[layer]), bits(outs_eager[layer])), f"layer {layer}"
    assert pa.device_error_flags() == 0
