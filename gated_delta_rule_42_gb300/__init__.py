"""GB300-native chunked KDA (Kimi Delta Attention): forward and backward for
training on sm_103a, behind a C-ABI library (``libkda.so``)."""
