"""The usage example the README quotes, run as written by the GPU tests."""
import torch
import server_side_fedavg_gb300 as fa

layout = [("embed", 32000 * 4096), ("lm_head", 32000 * 4096)]      # keys and their sizes
ctx = fa.fa_open(layout, "bf16", "bf16", max_clients=16)

# each client sends its update when it arrives; a client may send only some keys
upd = torch.empty(32000 * 4096, dtype=torch.bfloat16, device="cuda")   # client 0, key 0
fa.fa_accumulate(ctx, 0, 512.0, 0, 0, upd, upd.numel())              # weight = its sample count
host = torch.empty(32000 * 4096, dtype=torch.bfloat16).pin_memory()  # client 1, key 1, from host
fa.fa_accumulate(ctx, 1, 300.0, 1, 0, host, host.numel())            # read in place over the link

outs = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _, n in layout]
fa.fa_finalize(ctx, outs)          # per key: sum of n_k * w_k over the key's senders / their sum of n_k
fa.fa_sync(ctx)
fa.fa_reset(ctx)                   # next round; fa_close(ctx) when done
fa.fa_close(ctx)
