"""GB300-native Kimi Delta Attention (KDA): chunkwise prefill and recurrent decode.

The compute path is the CUDA C-ABI library built from csrc/ (see include/kda.h);
this package only marshals arguments into it.
"""
