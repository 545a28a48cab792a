"""GB300-native hyper-connection residual mixing."""
